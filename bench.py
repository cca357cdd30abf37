"""Benchmark of the TurboQuantProd hot path on B300: encode a KV cache, then score
one decode step on the compressed keys.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--bits B]

One step = tq_encode of every key of the workload (E0-E6) + tq_score of one
query per head against all of them (S0-S4).  The default workload is the
Qwen2.5-3B-shaped decode step (72 groups x 8,192 fp16 keys, 8 query heads per
group, d = 128, 3 bits).  The value is keys encoded-and-scored per second over
the whole step; the score-only and encode-only rates (``headline``),
per-kernel numbers, rooflines, the fp32-key baseline, an end-to-end run from
pinned host memory and the CPU oracle are reported beside it in the same JSON
line.  With the default workload the line also carries a score-only leg on the
other 3-bit d = 128 shape, the Llama-3.1-8B-shaped cache (4,096 groups x 32,768
bf16 keys, 4 heads per group), under ``parts.score_llama31_b3``.  Multi-GPU runs (torchrun) are replicas: every rank
runs the full workload on its own GPU (weak scaling), no collective on the
data path.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import tq_synth  # noqa: E402

METRIC = "tq_score keys scored/s & % HBM roofline at 3-bit d=128; tq_encode vectors/s"
DEFAULT_WORKLOAD = "qwen25_3b_decode"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
SPIN_CYCLES_PER_US = 2100  # at or above the maximum SM clock, so a spin lasts at least as long as asked
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


def kernel_traffic(kernel: str, source: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this workload and the current source of the kernel; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            tj = json.load(f)
        # an entry for this kernel on this workload, else the kernel's own
        t = tj.get(f"{kernel}@{workload}") or tj.get(kernel)
        with open(os.path.join(ROOT, "vector_quantization_02_b300", "csrc", source), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        if t and t.get("source_sha") == sha and t.get("workload") == workload:
            return t["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        pass
    return None


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region.
    A reader thread collects the rows; start() returns once the first sample
    has arrived, so that the region is covered from its beginning."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        import threading
        self.proc = None
        self.rows = []
        # nvidia-smi index of this CUDA device (CUDA_VISIBLE_DEVICES maps CUDA indices)
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        self.index = ids[device] if device < len(ids) and ids[device].isdigit() else str(device)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu=index,{self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.first = threading.Event()

        def read():
            for line in self.proc.stdout:
                if line.count(",") >= 8:
                    self.rows.append(line.strip().split(","))
                    self.first.set()
        self.thread = threading.Thread(target=read, daemon=True)
        self.thread.start()
        self.first.wait(timeout=15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.thread.join(timeout=10)
        rows = list(self.rows)
        if len({r[0].strip() for r in rows}) > 1:
            rows = [r for r in rows if r[0].strip() == self.index]
        rows = [r[1:] for r in rows]
        sm = [float(r[0]) for r in rows if r[0].strip().replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].strip() == "Active"})
        busy = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- oracle timing (CPU)

def oracle_throughput(w, bits, mode: str, budget_s: float, rotation: str = "dense"):
    """Time the oracle (encode + score of one group's keys against H heads) on a
    bounded sample; returns (keys/s, sample description, threads)."""
    import numpy as np

    from oracle import tq_oracle as o
    d = w.d
    if rotation == "hadamard":
        Pi = o.hadamard_rotation(tq_synth.hadamard_signs(d, w.seeds["rotation"]).double().numpy()).astype(np.float32)
    else:
        Pi = o.haar_rotation(tq_synth.rotation_gaussian(d, w.seeds["rotation"]).numpy()).astype(np.float32)
    S = tq_synth.projection(d, w.seeds["projection"]).numpy() if mode == "prod" else None
    c = o.codebook_f32(1 << (bits - 1 if mode == "prod" else bits), d)
    q = tq_synth.queries(w, G=1).numpy()

    def run(n):
        keys = tq_synth.keys(w, G=1, N=n)
        t0 = time.perf_counter()
        buf, _ = o.encode_pack(keys.double().numpy(), Pi, S, c, bits, mode, 1, n)
        o.score_packed(q, buf, Pi, S, c, bits, mode, 1, n)
        return time.perf_counter() - t0

    n = 256
    t = run(n)
    while t < budget_s / 8 and n < w.N:
        n = min(w.N, n * 4)
        t = run(n)
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except ImportError:
        threads = len(os.sched_getaffinity(0))
    return n / t, f"encode+score of {n} keys of group 0 against its {w.H} heads (numpy fp64)", threads


def workload_config(w, mode: str, bits: int, rotation: str = "dense") -> dict:
    """The workload as both arms report it."""
    return {"workload": w.name, "mode": mode, "G": w.G, "N": w.N, "H": w.H, "d": w.d, "bits": bits,
            "key_dtype": str(w.key_dtype).replace("torch.", ""), "top_k": w.top_k, "rotation": rotation}


# ---------------------------------------------------------------- our path

def roofline(bytes_, ms, kernel, source, workload, flops=None):
    """HBM roofline, or the bf16 tensor roofline where the algorithmic flops
    at that peak take longer than the bytes at HBM speed."""
    pk, pk_kind = peaks()
    hbm = pk["hbm_gbs"]
    tflops_peak = pk.get("bf16_tflops", FALLBACK_PEAKS.get("bf16_tflops"))
    ach = bytes_ / (ms * 1e-3) / 1e9
    tensor = flops is not None and flops / (tflops_peak * 1e12) > bytes_ / (hbm * 1e9)
    if tensor:
        tf = flops / (ms * 1e-3) / 1e12
        r = {"bound": "tensor", "achieved": round(tf, 2), "peak": tflops_peak, "unit": "TFLOP/s",
             "frac": round(tf / tflops_peak, 4)}
    else:
        r = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4)}
    r.update({"traffic": kernel_traffic(kernel, source, workload), "algorithmic_bytes": bytes_,
              "peak_source": pk_kind, "kernel": kernel})
    if flops is not None:
        r["algorithmic_flops"] = flops
        r["tflops"] = round(flops / (ms * 1e-3) / 1e12, 2)
        r["gbs"] = round(ach, 1)
    return r


def make_plan(w, bits: int, mode: str, rotation: str):
    """The workload's plan: the dense Haar rotation (QR of the seeded Gaussian)
    or the randomised Walsh-Hadamard rotation (signs seeded the same way)."""
    import vector_quantization_02_b300 as tq
    d = w.d
    S = None if mode == "mse" else tq_synth.projection(d, w.seeds["projection"])
    if rotation == "hadamard":
        k = bits - 1 if mode == "prod" else bits
        return tq.Plan.hadamard(d, bits, tq_synth.hadamard_signs(d, w.seeds["rotation"]), S,
                                tq.tq_lloyd_max_codebook(1 << k, d), mode=mode)
    return tq.Plan.from_seeds(d, bits, tq_synth.rotation_gaussian(d, w.seeds["rotation"]), S, mode=mode)


def encode_only_leg(w, bits: int, mode: str, rotation: str, keys, flush, reps: int, lead):
    """tq_encode alone on the step's keys with another plan (cold L2)."""
    import vector_quantization_02_b300 as tq
    plan = make_plan(w, bits, mode, rotation)
    G, N, d = keys.shape
    packed = torch.empty(plan.packed_bytes(G, N), dtype=torch.uint8, device=keys.device)
    stream = torch.cuda.current_stream()
    for _ in range(2):
        tq.tq_encode(plan, keys, packed=packed)
    times = []
    for _ in range(reps):
        flush.zero_()
        lead(300)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        tq.tq_encode(plan, keys, packed=packed)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    assert plan.status() == 0
    ms = statistics.median(a.elapsed_time(b) for a, b in times)
    kern = {"tensor_d128": ("encode_tc", "k_encode_tc.cu"), "tensor_wide": ("encode_wide", "k_encode_wide.cu")}
    kn, src = kern[plan.encode_path(w.key_dtype)]
    nbytes = keys.numel() * keys.element_size() + plan.packed_bytes(G, N)
    out = {"rotation": rotation, "ms_cold_l2": round(ms, 5), "vectors_per_s": G * N / (ms * 1e-3),
           "roofline_cold_l2": roofline(nbytes, ms, kn, src, w.name,
                                        flops=(2 if mode == "prod" else 1) * 2 * d * d * G * N), "reps": reps}
    plan.close()
    return out


def attend_leg(w, kplan, packed_k, q, flush, reps: int, lead):
    """tq_attend (one decode step of attention on the compressed cache) on the
    workload's keys and values drawn by the same generator (seed offset 7),
    values in a 3-bit TurboQuantMSE plan, scale 1/sqrt(d); cold L2."""
    import vector_quantization_02_b300 as tq
    G, N, H, d = w.G, w.N, w.H, w.d
    vbits = 3
    vplan = tq.Plan.from_seeds(d, vbits, tq_synth.rotation_gaussian(d, w.seeds["rotation"] + 1000), None, mode="mse")
    vals = tq_synth.keys(w, device=q.device, seed_offset=7)
    packed_v = tq.tq_encode_values(vplan, vals)
    del vals
    out = torch.empty(G, H, d, dtype=torch.float32, device=q.device)
    ws = torch.empty(tq.attend_workspace_bytes(kplan, vplan, G, H, N), dtype=torch.uint8, device=q.device)
    scale = 1.0 / d ** 0.5
    stream = torch.cuda.current_stream()
    for _ in range(2):
        tq.tq_attend(kplan, vplan, q, packed_k, packed_v, N, scale, out=out, workspace=ws)
    times = []
    for _ in range(reps):
        flush.zero_()
        lead(300)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        tq.tq_attend(kplan, vplan, q, packed_k, packed_v, N, scale, out=out, workspace=ws)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    assert kplan.status() == 0 and vplan.status() == 0
    ms = statistics.median(a.elapsed_time(b) for a, b in times)
    # algorithmic bytes: the packed keys and values once, queries in, outputs out
    nbytes = kplan.packed_bytes(G, N) + vplan.packed_bytes(G, N) + q.numel() * 4 + out.numel() * 4
    r = {"value_bits": vbits, "ms_cold_l2": round(ms, 5), "tokens_per_s": G * N / (ms * 1e-3),
         "roofline_cold_l2": roofline(nbytes, ms, "attend", "k_attend.cu", w.name),
         "launches": 4, "reps": reps,
         "note": "query preparation + score (logits to the workspace) + value contraction + split combine"}
    vplan.close()
    return r


def fractional_leg(w, keys, q, half_bits: int, flush, reps: int, lead):
    """Encode and score (cold L2) of the step's keys at a fractional width:
    half_bits / 2 bits per channel, the first d/2 rotated coordinates with
    one more Lloyd-Max bit (dense rotation of the workload's seed)."""
    import vector_quantization_02_b300 as tq
    G, N, H, d = w.G, w.N, w.H, w.d
    k_hi = (half_bits + 1) // 2 - 1
    Pi = tq.tq_haar_rotation(tq_synth.rotation_gaussian(d, w.seeds["rotation"]))
    plan = tq.Plan.fractional(d, half_bits, Pi, tq_synth.projection(d, w.seeds["projection"]),
                              tq.tq_lloyd_max_codebook(1 << k_hi, d), tq.tq_lloyd_max_codebook(1 << (k_hi - 1), d))
    packed = torch.empty(plan.packed_bytes(G, N), dtype=torch.uint8, device=q.device)
    logits = torch.empty(G, H, N, dtype=torch.float32, device=q.device)
    ws = torch.empty(tq.score_workspace_bytes(plan, G, H, N), dtype=torch.uint8, device=q.device)
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(2):
            fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            lead(300)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ts)

    enc_ms = timed(lambda: tq.tq_encode(plan, keys, packed=packed))
    sc_ms = timed(lambda: tq.tq_score(plan, q, packed, N, logits=logits, workspace=ws))
    assert plan.status() == 0
    P = plan.packed_bytes(G, N)
    out = {"bits_per_channel": half_bits / 2, "bytes_per_key": P // (G * (-(-N // 128)) * 128),
           "encode_ms_cold_l2": round(enc_ms, 5), "score_ms_cold_l2": round(sc_ms, 5),
           "encode_roofline_cold_l2": roofline(keys.numel() * keys.element_size() + P, enc_ms, "encode_tc",
                                               "k_encode_tc.cu", w.name, flops=2 * 2 * d * d * G * N),
           "score_roofline_cold_l2": roofline(P + G * H * N * 4 + q.numel() * 4, sc_ms, "score_tc", "k_score_tc.cu",
                                              w.name, flops=2 * 2 * d * H * G * N), "reps": reps}
    plan.close()
    return out


def score_only_leg(name: str, bits: int, flush, reps: int, dev, lead):
    """tq_score alone on a second workload, cold L2: the keys are encoded once,
    64 groups at a time (untimed), then one query per head is scored against
    every packed key.  Returns the leg's report."""
    import vector_quantization_02_b300 as tq
    w = tq_synth.WORKLOADS[name]
    G, N, H, d = w.G, w.N, w.H, w.d
    plan = tq.Plan.from_seeds(d, bits, tq_synth.rotation_gaussian(d, w.seeds["rotation"]),
                              tq_synth.projection(d, w.seeds["projection"]))
    per_group = plan.packed_bytes(1, N)
    packed = torch.empty(plan.packed_bytes(G, N), dtype=torch.uint8, device=dev)
    chunks = -(-G // tq_synth.KEY_CHUNK_GROUPS)
    for c in range(chunks):
        kc = tq_synth.key_chunk(w, c, device=dev)
        g0 = c * tq_synth.KEY_CHUNK_GROUPS
        tq.tq_encode(plan, kc, packed=packed[g0 * per_group:(g0 + kc.shape[0]) * per_group])
        del kc
    q = tq_synth.queries(w, device=dev)
    logits = torch.empty(G, H, N, dtype=torch.float32, device=dev)
    ws = torch.empty(tq.score_workspace_bytes(plan, G, H, N), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for _ in range(2):
        tq.tq_score(plan, q, packed, N, logits=logits, workspace=ws)
    times = []
    for _ in range(reps):
        flush.zero_()
        lead(300)
        a, b = ev(), ev()
        a.record(stream)
        tq.tq_score(plan, q, packed, N, logits=logits, workspace=ws)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    assert plan.status() == 0
    ms = statistics.median(a.elapsed_time(b) for a, b in times)
    P = plan.packed_bytes(G, N)
    sk = {"tensor_d128": ("score_tc", "k_score_tc.cu"), "tensor_wide": ("score_wide", "k_score_wide.cu")}
    kern, src = sk[plan.score_path(H)]
    out = {"workload": name, "bits": bits, "G": G, "N": N, "H": H, "d": d,
           "key_dtype": str(w.key_dtype).replace("torch.", ""), "ms_cold_l2": round(ms, 5),
           "keys_per_s_cold_l2": G * N / (ms * 1e-3), "logits_per_s_cold_l2": G * N * H / (ms * 1e-3),
           "roofline_cold_l2": roofline(P + G * H * N * 4 + q.numel() * 4, ms, kern, src, name,
                                        flops=2 * 2 * d * H * G * N),
           "launches": 2, "reps": reps}
    plan.close()
    del packed, logits, ws
    torch.cuda.empty_cache()
    return out

def _e2e(args, world, plan, keys, q, packed, logits, ws, flush, top_k, stream, ev):
    """Median step time with the inputs copied from pinned host memory and the
    logits copied back inside the timed events."""
    import vector_quantization_02_b300 as tq
    G, N, _ = keys.shape
    H = q.shape[1]
    keys_h = keys.cpu().pin_memory()
    q_h = q.cpu().pin_memory()
    out_h = torch.empty(G, H, N, dtype=torch.float32).pin_memory()
    keys_d = torch.empty_like(keys)
    q_d = torch.empty_like(q)
    e2e_t = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        a, b = ev(), ev()
        a.record(stream)
        keys_d.copy_(keys_h, non_blocking=True)
        q_d.copy_(q_h, non_blocking=True)
        tq.tq_encode(plan, keys_d, packed=packed)
        tq.tq_score(plan, q_d, packed, N, top_k=top_k, logits=logits, workspace=ws)
        out_h.copy_(logits, non_blocking=True)
        b.record(stream)
        if i >= args.warmup:
            e2e_t.append((a, b))
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, statistics.median(a.elapsed_time(b) for a, b in e2e_t))

    return e2e_ms


def workload(args):
    w = tq_synth.WORKLOADS[args.workload]
    if args.tokens:  # a reduced case of the same shape (profiling), never a bench value
        w = dataclasses.replace(w, N=min(args.tokens, w.N))
    return w


def run_ours(args, world, rank):
    import vector_quantization_02_b300 as tq
    w = workload(args)
    bits = args.bits or w.bits[0]
    dev = torch.device("cuda", torch.cuda.current_device())
    G, N, H, d = w.G, w.N, w.H, w.d

    keys = tq_synth.keys(w, device=dev, seed_offset=rank)
    q = tq_synth.queries(w, device=dev, seed_offset=rank)
    mse = args.mode == "mse"
    plan = make_plan(w, bits, args.mode, args.rotation)
    packed = torch.empty(plan.packed_bytes(G, N), dtype=torch.uint8, device=dev)
    logits = torch.empty(G, H, N, dtype=torch.float32, device=dev)
    top_k = w.top_k
    ws = torch.empty(tq.score_workspace_bytes(plan, G, H, N, top_k), dtype=torch.uint8, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * max(l2, 64 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        tq.tq_encode(plan, keys, packed=packed)
        tq.tq_score(plan, q, packed, N, top_k=top_k, logits=logits, workspace=ws)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def lead(us):
        # a device-side spin queued before a start event, outside the timed
        # region: the host enqueues the timed calls while it runs, so no
        # host launch gap falls between the events
        torch.cuda._sleep(int(us * SPIN_CYCLES_PER_US))

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    # clocks: the sampler is running (first sample in) before the timed region
    # starts and stops after a soak of the same step, so that its 100 ms samples
    # cover the timed steps even when they last a few milliseconds
    clocks = Clocks(dev.index)

    # timed region: K steps, L2 flushed between steps outside the step events
    e_start = [ev() for _ in range(args.steps)]
    e_mid = [ev() for _ in range(args.steps)]
    e_end = [ev() for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    lead(min(400 * args.steps, 100_000))
    for i in range(args.steps):
        flush.zero_()
        e_start[i].record(stream)
        tq.tq_encode(plan, keys, packed=packed)
        e_mid[i].record(stream)
        tq.tq_score(plan, q, packed, N, top_k=top_k, logits=logits, workspace=ws)
        e_end[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    soak_steps = 0
    while time.perf_counter() - t0 < args.soak_s:
        for _ in range(16):
            flush.zero_()
            step()
        soak_steps += 16
        torch.cuda.synchronize()
    clk = clocks.stop()
    clk["window"] = f"timed steps + {soak_steps} untimed steps of the same kind ({args.soak_s:.1f} s)"
    enc_ms = sum(a.elapsed_time(b) for a, b in zip(e_start, e_mid)) / args.steps
    sc_ms = sum(a.elapsed_time(b) for a, b in zip(e_mid, e_end)) / args.steps
    step_ms = max_over_ranks(world, enc_ms + sc_ms)
    assert plan.status() == 0
    keys_total = G * N * world
    value = keys_total / (step_ms * 1e-3)

    # per-kernel algorithmic bytes
    P = plan.packed_bytes(G, N)
    key_bytes = keys.numel() * keys.element_size()
    logit_bytes = G * H * N * 4
    q_bytes = q.numel() * 4
    enc_bytes = key_bytes + P
    sc_bytes = P + logit_bytes + q_bytes

    def roof(bytes_, ms, kernel, source, flops=None):
        return roofline(bytes_, ms, kernel, source, w.name, flops=flops)

    kernels = {"tensor_d128": ("{}_tc", "k_{}_tc.cu"), "tensor_wide": ("{}_wide", "k_{}_wide.cu")}
    ek, es = kernels[plan.encode_path(w.key_dtype)]
    enc_kernel, enc_src = ek.format("encode"), es.format("encode")
    # algorithmic flops: one d x d projection per key (Pi u), two in Prod (and S r)
    enc_roof = roof(enc_bytes, enc_ms, enc_kernel, enc_src,
                    flops=(2 if plan.mode == "prod" else 1) * 2 * d * d * G * N)

    # score alone on a cold L2 (a decode step reads a cache encoded earlier)
    sc_cold = []
    for _ in range(max(3, args.steps)):
        flush.zero_()
        lead(300)
        a, b = ev(), ev()
        a.record(stream)
        tq.tq_score(plan, q, packed, N, top_k=top_k, logits=logits, workspace=ws)
        b.record(stream)
        sc_cold.append((a, b))
    torch.cuda.synchronize()
    sc_cold_ms = statistics.median(a.elapsed_time(b) for a, b in sc_cold)
    sk, ss = kernels[plan.score_path(H)]
    arith = {"encode_tc": "f16/bf16 split operands on tensor cores",
             "encode_wide": "f16 split operands on tensor cores",
             "score_tc": "e4m3 bit planes and query slices on tensor cores", "score_wide":
             "bf16 split operands on tensor cores"}
    dtype_desc = (f"encode: {arith[enc_kernel]}; score: {arith[sk.format('score')]}; f32 accumulate")
    # algorithmic flops of the estimate: two length-d dot products per (key, head)
    sc_roof = roof(sc_bytes, sc_cold_ms, sk.format("score"), ss.format("score"),
                   flops=(2 if plan.mode == "prod" else 1) * 2 * d * H * G * N)

    # the uncompressed baseline on the same keys (fp32 copies), cold L2
    base = None
    if d * G * N * 4 < 40e9:
        keys32 = keys.float()
        base_l = torch.empty_like(logits)
        bt = []
        for _ in range(max(3, args.steps)):
            flush.zero_()
            lead(300)
            a, b = ev(), ev()
            a.record(stream)
            tq.tq_score_fp32(q, keys32, logits=base_l)
            b.record(stream)
            bt.append((a, b))
        torch.cuda.synchronize()
        bms = statistics.median(a.elapsed_time(b) for a, b in bt)
        base = {"ms": round(bms, 4), "keys_per_s": G * N / (bms * 1e-3),
                "roofline": roof(keys32.numel() * 4 + logit_bytes + q_bytes, bms, "score_fp32", "k_misc.cu",
                                 flops=2 * d * H * G * N),
                "score_speedup_vs_fp32_keys": round(bms / sc_cold_ms, 3)}
        del keys32, base_l

    # decode of every key (not part of the step), cold L2, on the tensor-core decode
    # of the plan's d (tensor_d128 or tensor_wide)
    dec = None
    dpath = plan.decode_path()
    if dpath in kernels and d * G * N * 4 < 40e9:
        xh = torch.empty(G, N, d, dtype=torch.float32, device=dev)
        dt = []
        for _ in range(max(3, args.steps)):
            flush.zero_()
            lead(300)
            a, b = ev(), ev()
            a.record(stream)
            tq.tq_decode(plan, packed, G, N, out=xh)
            b.record(stream)
            dt.append((a, b))
        torch.cuda.synchronize()
        assert plan.status() == 0
        dms = statistics.median(a.elapsed_time(b) for a, b in dt)
        # algorithmic bytes: the packed keys in, fp32 rows out; flops: one d x d
        # product per key, two in Prod
        dec = {"ms": round(dms, 5), "vectors_per_s": G * N / (dms * 1e-3),
               "roofline": roof(P + G * N * d * 4, dms, kernels[dpath][0].format("decode"),
                                kernels[dpath][1].format("decode"),
                                flops=(2 if plan.mode == "prod" else 1) * 2 * d * d * G * N)}
        del xh

    # one decode step of attention on the same compressed keys and values
    att = None
    if d == 128 and args.mode == "prod" and not mse:
        try:
            att = attend_leg(w, plan, packed, q, flush, max(5, args.steps), lead)
        except tq.TQError:
            att = None  # a shape tq_attend does not take

    # the same keys at a fractional width (3.5 bits per channel)
    frac = None
    if d == 128 and args.mode == "prod" and w.key_dtype != torch.float32 and H <= 16:
        frac = fractional_leg(w, keys, q, 7, flush, max(5, args.steps), lead)

    # the same encode with the randomised Walsh-Hadamard rotation (or, when the
    # step itself uses it, with the dense rotation)
    other = "dense" if args.rotation == "hadamard" else "hadamard"
    enc_other = None
    if (d & (d - 1)) == 0:
        enc_other = encode_only_leg(w, bits, args.mode, other, keys, flush, max(5, args.steps), lead)

    # end to end through the public API from pinned host memory
    if key_bytes > 8e9:
        e2e_ms = None
    else:
        e2e_ms = _e2e(args, world, plan, keys, q, packed, logits, ws, flush, top_k, stream, ev)
    # our kernels per step: the encode (encode_tc_kernel, or key_norm_kernel +
    # encode_wide_kernel), the score (score_tc_prep_kernel + score_tc_kernel, or
    # the query projections + wide_split_kernel + score_wide_kernel) and top-k
    enc_launches = 1 if plan.encode_path(w.key_dtype) == "tensor_d128" else 2
    sc_launches = 2 if plan.score_path(H) == "tensor_d128" else 3
    launches_per_step = enc_launches + sc_launches + (2 if top_k else 0)
    line = {
        "metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype_desc,
        "data": "synthetic",
        "config": workload_config(w, args.mode, bits, args.rotation),
        "l2": "flushed between steps (2x L2 memset, outside the step events)",
        "headline": {
            "step_keys_per_s": value,
            "score_keys_per_s_cold_l2": G * N / (sc_cold_ms * 1e-3), "score_hbm_frac": sc_roof["frac"],
            "encode_vectors_per_s": G * N / (enc_ms * 1e-3), "encode_roofline_frac": enc_roof["frac"],
            "note": "value = keys encoded and scored per second over the whole step (encode + score); the "
                    "score-only and encode-only rates are given here and under parts"},
        "roofline": enc_roof,
        "parts": {
            "encode": {"ms": round(enc_ms, 5), "vectors_per_s": G * N / (enc_ms * 1e-3), "roofline": enc_roof},
            "score": {"ms_in_step": round(sc_ms, 5), "ms_cold_l2": round(sc_cold_ms, 5),
                      "keys_per_s_cold_l2": G * N / (sc_cold_ms * 1e-3),
                      "logits_per_s_cold_l2": G * N * H / (sc_cold_ms * 1e-3), "roofline_cold_l2": sc_roof},
            "fp32_key_baseline": base,
            "decode": dec,
            f"encode_{other}": enc_other,
            "attend": att,
            "fractional_3p5": frac,
        },
        "e2e": None if e2e_ms is None else {
            "value": keys_total / (e2e_ms * 1e-3), "unit": "keys/s", "h2d_bytes_per_step": key_bytes + q_bytes,
            "d2h_bytes_per_step": logit_bytes, "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 4),
    }
    plan.close()
    if args.second_leg and args.workload == DEFAULT_WORKLOAD and args.mode == "prod" and not args.tokens:
        # the other 3-bit d = 128 headline shape: score alone on the Llama-3.1-8B cache
        del keys, packed, logits, ws
        torch.cuda.empty_cache()
        line["parts"]["score_llama31_b3"] = score_only_leg("llama31_8b_prefill", 3, flush, max(5, args.steps), dev,
                                                           lead)
    if rank == 0 and not args.no_cpu_baseline:
        v, sample, cores = oracle_throughput(w, bits, args.mode, args.cpu_budget, args.rotation)
        line["cpu_baseline"] = {"value": v, "unit": "keys/s", "cores": cores, "kind": "oracle", "sample": sample}
    return line


def run_reference(args, world, rank):
    w = workload(args)
    bits = args.bits or w.bits[0]
    if rank != 0:
        return None
    vals = []
    sample = cores = None
    for _ in range(args.warmup + args.steps):
        v, sample, cores = oracle_throughput(w, bits, args.mode, args.cpu_budget / max(1, args.steps + args.warmup),
                                             args.rotation)
        vals.append(v)
    v = statistics.median(vals[args.warmup:]) if len(vals) > args.warmup else vals[-1]
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "keys/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.mode, bits, args.rotation),
        "cpu_baseline": {"value": v, "unit": "keys/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "keys/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(tq_synth.WORKLOADS))
    ap.add_argument("--bits", type=int, default=0)
    ap.add_argument("--mode", choices=["prod", "mse"], default="prod",
                    help="TurboQuantProd (the workloads' method) or TurboQuantMSE codec")
    ap.add_argument("--rotation", choices=["dense", "hadamard"], default="dense",
                    help="dense Haar rotation (QR of a seeded Gaussian) or randomised Walsh-Hadamard rotation")
    ap.add_argument("--tokens", type=int, default=0,
                    help="cap the tokens per group (a reduced case for profiling; not a bench configuration)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-second-leg", dest="second_leg", action="store_false",
                    help="skip the score-only leg on the Llama-3.1-8B-shaped cache at 3 bits")
    ap.add_argument("--soak-s", type=float, default=1.5,
                    help="seconds (from the start of the timed region) the step keeps running while clocks are sampled")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, _ = dist_setup(args)
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_ours(args, world, rank)
    if rank == 0 and line is not None:
        if args.tokens and "config" in line:
            line["config"]["reduced_for_profiling"] = True
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
