#!/usr/bin/env python
"""Benchmark of the Q8_0 Llama forward on GB300.

Workload (one "step"): the 135M-shaped Q8_0 Llama with random weights
(seed 0), a fresh KV cache, one 203-token prefill of uniform random ids, then
128 greedy decode steps — the task of the candle page "速度"
(两边量的是同一件事: 203-token prefill + 128 greedy decode steps, repeated
with a fresh cache). The headline metric is decode tokens/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl ours (default): the CUDA library; device-timed with CUDA events on the
library's stream, inputs resident in HBM; plus an end-to-end number through
the host API, per-kernel timing, the 7B-shape GEMV roofline and the CPU
oracle baseline. --impl reference: the CPU oracle on this host's cores on the
same workload, each step a bounded sample (prefill + a few decode steps).
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the model does not shard); rank 0 prints one JSON line.
"""
from __future__ import annotations

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

METRIC = "decode tokens/s + ms/token; Q8_0 GEMV HBM GB/s vs peak (Q8_0 Llama, 1 GB300)"
PROMPT_LEN = 203
DECODE_STEPS = 128
SEED = 0
# The pages' number for this task and metric: Q8_0 decode 7.40 ms/token on an
# M2 Max CPU ("速度", CPU GGUF：decode 快，prefill 慢). Context, not the target.
PAGES_DECODE_MS = 7.40
FALLBACK_HBM_GBS = 6800.0
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# decode step's kernels from one ncu capture of the current kernel sources
# (135M model, decode steps after the 203-token prompt, kv_len stated); the
# K/V part grows by n_kv * head_dim * 8 bytes per cached position.
NCU_TRAFFIC = {
    # 3 launches (layers 0-2 of decode step 21, kv_len 224), mean of 1,344,768 / 1,358,592 / 1,358,336 B read, 0 written
    "layer_front_qkv_attn_o": {"bytes": 1353899, "kv_len": 224, "kv_bytes_per_pos": 1536},
}
FP32_FMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12  # SMs x FP32 lanes x 2 flops x max SM clock
L2_BYTES = 126 * 2 ** 20


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--cpu-baseline-seconds", type=float, default=20.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-baseline-worker", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--cpu-baseline-threads", type=int, default=0, help=argparse.SUPPRESS)
    p.add_argument("--cpu-baseline-config", choices=["c0", "c1", "c4"], default="c1", help=argparse.SUPPRESS)
    p.add_argument("--only", choices=["gemv7b", "formats", "attn", "gemm", "decode", "decode7b", "prefill",
                                      "prefill7b", "sweep", "attnprefill", "profile"],
                   default=None,
                   help="run one kernel workload only (used for ncu captures)")
    return p.parse_args(argv)


# ----------------------------------------------------------------------------
# multi-rank plumbing (replicas)
# ----------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (x itself at world == 1)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, elapsed_s: float, world: int, device=None) -> tuple[float, float]:
    """Whole-job throughput: units of all ranks / the slowest rank's time."""
    t = max_over_ranks(elapsed_s, world, device)
    return units_per_rank * world / t, t


# ----------------------------------------------------------------------------
# peaks and clocks
# ----------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for key in ("hbm_gbs", "hbm_GBps", "hbm"):
                if key in d:
                    v = d[key]
                    return float(v["value"] if isinstance(v, dict) else v), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"lq8_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        try:
            self.fh.close()
        except Exception:
            pass

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# CPU oracle legs
# ----------------------------------------------------------------------------

def oracle_model(big: bool = False):
    """The oracle's model: the 135M shape (seed 0), or the 7B shape (seed 1)."""
    from oracle import q8_oracle as O
    from q8_quantized_llama_gb300 import synth
    cfg = dict(synth.MODEL_7B if big else synth.MODEL_135M)
    t = {}
    for name, w, kind in synth.iter_model_weights_f32(cfg, 1 if big else SEED):
        t[name] = O.quantize_q8_0(w) if kind == "matrix" else w
    return O, cfg, O.ModelWeights(cfg, t, weight_cache="f64")


def oracle_step(O, model, prompt, n_decode):
    """Prefill + n_decode greedy steps on the oracle; returns (prefill_s, decode_s)."""
    t0 = time.perf_counter()
    logits = model.forward(prompt, 0)
    t1 = time.perf_counter()
    nxt = O.argmax_lowest(logits)
    pos = len(prompt)
    for _ in range(n_decode):
        nxt = O.argmax_lowest(model.forward([nxt], pos))
        pos += 1
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def cpu_threads() -> int:
    return os.cpu_count() or 1


# The oracle's configurations: model, prompt length, decode steps of the full
# run, and the decode steps of the bounded sample (C4: prefill + the first 16
# decode steps; the full 256 would take far longer than a bench run).
ORACLE_CONFIGS = {
    "c0": (False, 13, 20, 20),
    "c1": (False, PROMPT_LEN, DECODE_STEPS, DECODE_STEPS),
    "c4": (True, 512, 256, 16),
}


def cpu_baseline_worker(seconds: float, threads: int = 0, config: str = "c1"):
    """Runs in a fresh interpreter: the oracle on a bounded sample of one
    configuration (threads > 0: the BLAS/OpenMP thread count the parent set)."""
    from q8_quantized_llama_gb300 import synth
    big, n_prompt, n_full, n_sample = ORACLE_CONFIGS[config]
    O, cfg, model = oracle_model(big)
    prompt = synth.prompt_ids(n_prompt, cfg["n_vocab"], 1 if big else SEED)
    t_start = time.perf_counter()
    t0 = time.perf_counter()
    nxt = O.argmax_lowest(model.forward(prompt, 0))
    p_s = time.perf_counter() - t0
    pos, n, d_s = n_prompt, 0, 0.0
    while n < n_sample and time.perf_counter() - t_start < seconds:
        t0 = time.perf_counter()
        nxt = O.argmax_lowest(model.forward([nxt], pos))
        d_s += time.perf_counter() - t0
        pos += 1
        n += 1
    name = "7B" if big else "135M"
    print(json.dumps({"value": n / d_s if n else None, "unit": "tokens/s", "cores": threads or cpu_threads(),
                      "kind": "oracle", "config": config, "prefill_tok_s": n_prompt / p_s,
                      "decode_ms_per_token": 1000 * d_s / n if n else None,
                      "sample": f"{name} Q8_0 oracle (numpy f64): one {n_prompt}-token prefill and the first {n} "
                                f"of the {n_full} greedy decode steps"}))


def run_cpu_baseline(seconds: float, threads: int = 0, config: str = "c1", timeout: float = 600.0):
    """The oracle timed in a subprocess on all host cores, or (threads > 0) with
    the BLAS and OpenMP pools held to that many threads."""
    env = dict(os.environ)
    if threads > 0:
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
            env[var] = str(threads)
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-worker",
                            "--cpu-baseline-seconds", str(seconds), "--cpu-baseline-threads", str(threads),
                            "--cpu-baseline-config", config],
                           capture_output=True, text=True, env=env, timeout=timeout)
    except subprocess.TimeoutExpired:
        return {"value": None, "unit": "tokens/s", "cores": threads or cpu_threads(), "kind": "oracle",
                "config": config, "sample": f"not finished within {timeout:.0f} s"}
    for line in r.stdout.splitlines()[::-1]:
        if line.startswith("{"):
            return json.loads(line)
    return {"value": None, "unit": "tokens/s", "cores": threads or cpu_threads(), "kind": "oracle",
            "config": config, "sample": "failed: " + r.stderr[-300:]}


def run_reference(args):
    """The oracle as it stands on the workload of the headline metric: each
    step one 203-token prefill and all 128 greedy decode steps (decode
    tokens/s over the timed steps)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from q8_quantized_llama_gb300 import synth
    O, cfg, model = oracle_model()
    prompt = synth.prompt_ids(PROMPT_LEN, cfg["n_vocab"], SEED)
    n_dec = DECODE_STEPS
    for _ in range(args.warmup):
        oracle_step(O, model, prompt, n_dec)
    pre, dec = [], []
    for _ in range(args.steps):
        p_s, d_s = oracle_step(O, model, prompt, n_dec)
        pre.append(p_s)
        dec.append(d_s)
    value = n_dec * args.steps / sum(dec)
    sample = (f"135M Q8_0 oracle (numpy f64), each step the whole workload: one 203-token prefill + all "
              f"{n_dec} greedy decode steps")
    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": 1000 * (sum(pre) + sum(dec)) / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": {"workload": "135M-shaped Q8_0 Llama (30x576, 9/3 heads, FFN 1536, vocab 49152, seed 0): "
                                  "203-token random prompt prefill + 128 greedy decode steps, fresh KV cache",
                      "prompt": PROMPT_LEN, "decode_steps": n_dec},
           "decode_ms_per_token": 1000 * sum(dec) / (n_dec * args.steps),
           "prefill_tok_s": PROMPT_LEN * args.steps / sum(pre),
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def gpu_model(torch, B, synth, device, head_splits=0):
    cfg = dict(synth.MODEL_135M, head_splits=head_splits)
    t = {}
    for name, w, kind in synth.iter_model_weights_f32(cfg, SEED):
        dw = torch.from_numpy(w).to(device)
        if kind == "matrix":
            q = torch.empty((w.shape[0], w.shape[1] // 32 * 34), dtype=torch.uint8, device=device)
            B.llama_q8_quantize(dw, w.shape[0], w.shape[1], q, torch.cuda.current_stream().cuda_stream)
            t[name] = q
        else:
            t[name] = dw
    torch.cuda.synchronize()
    model = B.Model(cfg, t, device=device.index, on_device=True)
    del t
    torch.cuda.empty_cache()
    return cfg, model


def q8_bytes(rows: int, k: int) -> float:
    return rows * k * 34 / 32


def decode_bytes(cfg: dict, kv_len: float) -> tuple[float, float]:
    """Algorithmic bytes of one decode step: (Q8_0 weights of every projection
    and the lm_head + f32 norms, f32 K and V rows read by the attention)."""
    h, hd, F = cfg["n_embd"], cfg["head_dim"], cfg["n_ff"]
    qd, kvd = cfg["n_head"] * hd, cfg["n_head_kv"] * hd
    per_layer = q8_bytes(qd + 2 * kvd, h) + q8_bytes(h, qd) + q8_bytes(2 * F, h) + q8_bytes(h, F) + 8 * h
    weights = cfg["n_layer"] * per_layer + q8_bytes(cfg["n_vocab"], h) + 4 * h + q8_bytes(1, h)
    kv = 2 * cfg["n_layer"] * kvd * 4 * kv_len
    return weights, kv


def gpu_model_7b(torch, B, synth, device):
    """The Llama-7B-shaped Q8_0 model: weights N(0, 0.02) drawn on the GPU
    (seed 1) and quantised there, norm weights 1 + N(0, 0.02)."""
    cfg = dict(synth.MODEL_7B)
    gen = torch.Generator(device=device)
    gen.manual_seed(1)
    t = {}
    s = torch.cuda.current_stream()
    for name, shape, kind in synth.model_tensor_specs(cfg):
        if kind == "matrix":
            rows, k = shape
            w = torch.randn(shape, generator=gen, device=device) * synth.WEIGHT_STD
            q = torch.empty((rows, k // 32 * 34), dtype=torch.uint8, device=device)
            B.llama_q8_quantize(w, rows, k, q, s.cuda_stream)
            del w
            t[name] = q
        else:
            t[name] = 1.0 + synth.WEIGHT_STD * torch.randn(shape, generator=gen, device=device)
    torch.cuda.synchronize()
    model = B.Model(cfg, t, device=device.index, on_device=True)
    del t
    torch.cuda.empty_cache()
    return cfg, model


def prefill_only(torch, B, synth, device, args, big: bool):
    """Prefill alone (the 203-token prompt on the 135M model, or 512 tokens on
    the 7B model), W warm-up and K timed calls on the library stream: the
    command behind the prefill launch lists."""
    cfg, model = gpu_model_7b(torch, B, synth, device) if big else gpu_model(torch, B, synth, device)
    n = 512 if big else PROMPT_LEN
    prompt = synth.prompt_ids(n, cfg["n_vocab"], 1 if big else SEED)
    d_prompt = torch.from_numpy(prompt).to(device)
    d_next = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.ExternalStream(model.stream(), device=device)
    for _ in range(max(1, args.warmup)):
        model.prefill_async(d_prompt, n, 0, d_next)
    model.sync()
    l0 = model.launch_count()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    torch.cuda.nvtx.range_push("timed_region")
    for i in range(args.steps):
        ev[i][0].record(stream)
        model.prefill_async(d_prompt, n, 0, d_next)
        ev[i][1].record(stream)
    model.sync()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    ms = [e[0].elapsed_time(e[1]) for e in ev]
    out = {"workload": f"{'7B' if big else '135M'}-shaped Q8_0 Llama, {n}-token prefill",
           "prefill_ms": statistics.median(ms), "prefill_tok_s": n / (statistics.median(ms) / 1000),
           "launches_per_prefill": (model.launch_count() - l0) / args.steps}
    model.close()
    return out


def decode_7b(torch, B, synth, device, peak, prompt_len=512, n_decode=256, reps=3):
    """Greedy decode of the Llama-7B-shaped Q8_0 model (32 x 4096, 32/8 heads of
    128, FFN 14336, vocab 32000, untied head) after a 512-token prefill: the
    decode step streams 7.55 GB of weights, so this is where the matrix-vector
    kernel's bandwidth shows in a whole model. Weights N(0, 0.02) drawn on the
    GPU (seeded) and quantised there; ms/token timed with CUDA events on the
    library stream over the CUDA-graph decode steps."""
    cfg, model = gpu_model_7b(torch, B, synth, device)
    prompt = synth.prompt_ids(prompt_len, cfg["n_vocab"], 1)
    d_prompt = torch.from_numpy(prompt).to(device)
    d_next = torch.zeros(1, dtype=torch.int32, device=device)
    d_out = torch.zeros(n_decode, dtype=torch.int32, device=device)
    stream = torch.cuda.ExternalStream(model.stream(), device=device)
    model.prefill_async(d_prompt, prompt_len, 0, d_next)
    model.decode_async(8, d_out)
    model.sync()
    pre, dec = [], []
    for rep in range(reps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        model.prefill_async(d_prompt, prompt_len, 0, d_next)
        e[1].record(stream)
        if rep == 0:
            torch.cuda.nvtx.range_push("timed_region")  # the decode steps (launch-list captures)
        model.decode_async(n_decode, d_out)
        if rep == 0:
            torch.cuda.nvtx.range_pop()
        e[2].record(stream)
        model.sync()
        torch.cuda.synchronize()
        pre.append(e[0].elapsed_time(e[1]))
        dec.append(e[1].elapsed_time(e[2]) / n_decode)
    # per-kernel in-graph times: the instrumented graph over 64 steps after the prompt
    model.prefill_async(d_prompt, prompt_len, 0, d_next)
    model.sync()
    fams, prof_step_us = decode_timeline(model, cfg, 64, peak)
    model.close()
    torch.cuda.empty_cache()
    ms = statistics.median(dec)
    w, kv = decode_bytes(cfg, prompt_len + (n_decode + 1) / 2)
    roof_ms = (w + kv) / (peak * 1e9) * 1e3
    return {"workload": f"7B-shaped Q8_0 Llama, {prompt_len}-token prefill + {n_decode} greedy decode steps",
            "decode_ms_per_token": ms, "decode_tok_s": 1000.0 / ms, "prefill_ms": statistics.median(pre),
            "prefill_tok_s": prompt_len / (statistics.median(pre) / 1000),
            "weights_bytes": w, "kv_bytes_mean": kv, "roofline_ms": roof_ms, "frac": roof_ms / ms,
            "instrumented_step_us": prof_step_us, "kernels": fams}


def gemv_7b_roofline(torch, B, synth, device, peak):
    """The Q8_0 GEMV at the 7B shape [1,4096]x[4096,14336], timed with CUDA
    events over 400 back-to-back launches that rotate through 8 weight copies
    (8 x 62.4 MB > L2), so every launch streams its matrix from HBM. Two forms:
    "chained" lets each launch start its weight stream while the previous one
    finishes (the way the decode step chains its projections), "serial" waits
    for the previous launch to end before the next one starts."""
    rows, k = 14336, 4096
    w = synth.weight_matrix_f32(rows, k, 1)
    dw = torch.from_numpy(w).to(device)
    q = torch.empty((rows, k // 32 * 34), dtype=torch.uint8, device=device)
    B.llama_q8_quantize(dw, rows, k, q)
    nbytes = B.llama_q8_packed_bytes(rows, k)
    copies = [torch.empty(nbytes, dtype=torch.uint8, device=device) for _ in range(8)]
    for c in copies:
        B.llama_q8_pack(q, rows, k, c)
    del dw, q
    x = torch.from_numpy(synth.normal_f32((1, k), 1, 7)).to(device)
    y = torch.empty((1, rows), dtype=torch.float32, device=device)
    s = torch.cuda.current_stream()
    algo = rows * k * 34 / 32 + 4 * k + 4 * rows
    res = {}
    for form, flags in (("serial", 0), ("chained", B.LQ8_MATMUL_EARLY_WEIGHTS)):
        for i in range(16):
            B.llama_q8_matmul_ex(copies[i % 8], rows, k, x, 1, y, flags, s.cuda_stream)
        n = 400
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s)
        for i in range(n):
            B.llama_q8_matmul_ex(copies[i % 8], rows, k, x, 1, y, flags, s.cuda_stream)
        e1.record(s)
        torch.cuda.synchronize()
        res[form] = e0.elapsed_time(e1) * 1000 / n
    del copies
    torch.cuda.empty_cache()
    us = res["chained"]
    gbs = algo / (us * 1e-6) / 1e9
    return {"kernel": "q8_gemv_kernel<EPI_STORE>", "shape": "[1,4096]x[4096,14336]", "us": us,
            "form": "chained launches (weight stream starts before the previous launch ends)",
            "algorithmic_bytes": algo, "achieved_gbs": gbs, "peak_gbs": peak, "frac": gbs / peak,
            "serial_us": res["serial"], "serial_frac": algo / (res["serial"] * 1e-6) / 1e9 / peak}


def block_format_gemv_bench(torch, B, synth, device, peak):
    """The matrix-vector product in the other GGUF block formats of a Q4_K_M
    file ("速度", CPU GGUF：decode 快，prefill 慢: Q5_0, Q4K, Q6K), with Q8_0
    beside them, at two shapes: [1,4096]x[4096,14336] for bandwidth (chained
    launches rotating over 8 weight copies, 8 x 33-62 MB > L2, so each launch
    streams its matrix from HBM) and the pages' QMatMul shape
    [1,1536]x[1536,576] (latency bound; 64 rotating copies). Algorithmic bytes
    = rows * k * (block bytes / block weights) + 4 k + 4 rows."""
    formats = (("Q8_0", B.GGUF_Q8_0, 34 / 32), ("Q5_0", B.GGUF_Q5_0, 22 / 32), ("Q4_K", B.GGUF_Q4_K, 144 / 256),
               ("Q6_K", B.GGUF_Q6_K, 210 / 256))
    s = torch.cuda.current_stream()
    out = []
    for rows, k, ncopy, n in ((14336, 4096, 8, 200), (576, 1536, 64, 400)):
        x = torch.from_numpy(synth.normal_f32((1, k), 3, 7)).to(device)
        y = torch.empty((1, rows), dtype=torch.float32, device=device)
        for name, t, bpw in formats:
            if t == B.GGUF_Q8_0:
                w = torch.from_numpy(synth.weight_matrix_f32(rows, k, 3)).to(device)
                blob = torch.empty((rows, k // 32 * 34), dtype=torch.uint8, device=device)
                B.llama_q8_quantize(w, rows, k, blob)
                del w
            else:
                blob = torch.from_numpy(synth.random_blocks(t, rows, k, 3)).to(device)
            nbytes = B.llama_q8_packed_bytes_fmt(t, rows, k)
            first = torch.empty(nbytes, dtype=torch.uint8, device=device)
            B.llama_q8_pack_fmt(t, blob, rows, k, first)
            del blob
            copies = [first] + [first.clone() for _ in range(ncopy - 1)]
            flags = B.LQ8_MATMUL_EARLY_WEIGHTS
            for i in range(16):
                B.llama_q8_matvec_fmt(t, copies[i % ncopy], rows, k, x, y, flags, s.cuda_stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(s)
            for i in range(n):
                B.llama_q8_matvec_fmt(t, copies[i % ncopy], rows, k, x, y, flags, s.cuda_stream)
            e1.record(s)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1000 / n
            algo = rows * k * bpw + 4 * k + 4 * rows
            gbs = algo / (us * 1e-6) / 1e9
            out.append({"format": name, "shape": f"[1,{k}]x[{k},{rows}]", "us": us, "algorithmic_bytes": algo,
                        "achieved_gbs": gbs, "frac": gbs / peak})
            del copies, first
            torch.cuda.empty_cache()
    return out


def gemm_microbench(torch, B, synth, device):
    """Q8_0 matrix-matrix products: the pages' QMatMul
    shape [203,1536]x[1536,576] ("速度", CPU GGUF), the 135M prefill shapes at
    203 rows, and 7B prefill shapes at 512 rows, with the library's choice of
    kernel and with each kernel forced (tensor cores, CUDA-core rows kernel).
    Algorithmic TFLOP/s = 2*m*rows*k / time of the automatic choice."""
    out = []
    s = torch.cuda.current_stream()
    for m, rows, k in ((203, 576, 1536), (203, 960, 576), (203, 3072, 576), (512, 6144, 4096), (512, 28672, 4096),
                       (512, 4096, 14336)):
        w = synth.weight_matrix_f32(rows, k, 5, stream=rows + k)
        dw = torch.from_numpy(w).to(device)
        q = torch.empty((rows, k // 32 * 34), dtype=torch.uint8, device=device)
        B.llama_q8_quantize(dw, rows, k, q)
        packed = torch.empty(B.llama_q8_packed_bytes(rows, k), dtype=torch.uint8, device=device)
        B.llama_q8_pack(q, rows, k, packed)
        del dw, q
        x = torch.from_numpy(synth.normal_f32((m, k), 5, 1)).to(device)
        y = torch.empty((m, rows), dtype=torch.float32, device=device)
        rec = {"shape": f"[{m},{k}]x[{k},{rows}]"}
        # the automatic choice first, then each kernel forced by flag
        for key, flags in (("auto", 0), ("tensor_cores", B.LQ8_MATMUL_TENSOR_CORES),
                           ("cuda_cores", B.LQ8_MATMUL_CUDA_CORES)):
            for _ in range(3):
                B.llama_q8_matmul_ex(packed, rows, k, x, m, y, flags, s.cuda_stream)
            n = 20
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(n):
                B.llama_q8_matmul_ex(packed, rows, k, x, m, y, flags, s.cuda_stream)
            e1.record(s)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1000 / n
            if key == "auto":
                rec.update({"us": us, "tflops": 2.0 * m * rows * k / (us * 1e-6) / 1e12})
            else:
                rec[key + "_us"] = us
        out.append(rec)
        del packed, x, y
        torch.cuda.empty_cache()
    return out


def linear_sweep(torch, B, synth, device, peak):
    """The Q8_0 linear sweep: x [rows, K] (N(0,1) f32) times each 135M
    projection shape at rows 1, 8 and 203 — [576->576] (q, o), [576->192]
    (k, v), [576->1536] (gate, up), [1536->576] (down), [576->49152] (lm_head)
    — plus the 7B shapes [1,4096]x[4096,4096] and x[4096,14336]. Each timed
    launch reads its own copy of the weights, rotating over enough copies to
    exceed L2 (>= 256 MB), so the weights stream from HBM; rows = 1 launches
    are chained the way the decode step chains them. GB/s counts the algorithmic
    bytes (N*K*34/32 + 4*K*rows + 4*N*rows); rows = 203 also TFLOP/s."""
    out = []
    s = torch.cuda.current_stream()
    shapes = [(r, n, k) for r in (1, 8, 203) for n, k in ((576, 576), (192, 576), (1536, 576), (576, 1536),
                                                            (49152, 576))]
    shapes += [(1, 4096, 4096), (1, 14336, 4096)]
    for rows, n, k in shapes:
        w = synth.weight_matrix_f32(n, k, 9, stream=n + k)
        dw = torch.from_numpy(w).to(device)
        q = torch.empty((n, k // 32 * 34), dtype=torch.uint8, device=device)
        B.llama_q8_quantize(dw, n, k, q)
        nbytes = B.llama_q8_packed_bytes(n, k)
        ncopy = max(2, min(1024, -(-256 * 2 ** 20 // nbytes)))
        packed = torch.empty((ncopy, nbytes), dtype=torch.uint8, device=device)
        for c in range(ncopy):
            B.llama_q8_pack(q, n, k, packed[c])
        del dw, q
        x = torch.from_numpy(synth.normal_f32((rows, k), 9, 2)).to(device)
        y = torch.empty((rows, n), dtype=torch.float32, device=device)
        flags = B.LQ8_MATMUL_EARLY_WEIGHTS if rows == 1 else 0
        launches = max(ncopy, 200) if rows == 1 else max(ncopy, 50)
        for i in range(min(ncopy, 16)):
            B.llama_q8_matmul_ex(packed[i], n, k, x, rows, y, flags, s.cuda_stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s)
        for i in range(launches):
            B.llama_q8_matmul_ex(packed[i % ncopy], n, k, x, rows, y, flags, s.cuda_stream)
        e1.record(s)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1000 / launches
        algo = n * k * 34 / 32 + 4 * k * rows + 4 * n * rows
        rec = {"shape": f"[{rows},{k}]x[{k},{n}]", "us": us, "gbs": algo / (us * 1e-6) / 1e9,
               "frac": algo / (us * 1e-6) / 1e9 / peak, "weight_copies": ncopy}
        if rows == 203:
            rec["tflops"] = 2.0 * rows * n * k / (us * 1e-6) / 1e12
        out.append(rec)
        del packed, x, y
        torch.cuda.empty_cache()
    return out


def attention_prefill_bench(torch, B, synth, device):
    """Causal prefill attention (llama_q8_attention, T > 1): T = 203 at
    position 0, T = 64 at position 512 and T = 512 at position 0 (the 7B
    prefill's length), at the 135M shape (9/3 heads of 64)
    and the 7B shape (32/8 heads of 128), cache stride 4096. Algorithmic
    FLOP = 4 * n_head * head_dim * sum over queries of the visible positions
    (q k^T and p v); the kernel runs on the FP32 CUDA cores, so the fraction is
    of the FP32 FMA rate at the maximum SM clock."""
    out = []
    s = torch.cuda.current_stream()
    for nh, nkv, hd in ((9, 3, 64), (32, 8, 128)):
        stride = 4096
        kc = torch.from_numpy(synth.normal_f32((nkv, stride, hd), 3, 1)).to(device)
        vc = torch.from_numpy(synth.normal_f32((nkv, stride, hd), 3, 2)).to(device)
        for T, pos in ((203, 0), (64, 512), (512, 0)):
            q = torch.from_numpy(synth.normal_f32((T, nh, hd), 3, 3)).to(device)
            o = torch.empty((T, nh, hd), dtype=torch.float32, device=device)
            for _ in range(3):
                B.llama_q8_attention(q, kc, vc, T, pos, nh, nkv, hd, stride, o, None, 0, s.cuda_stream)
            n = 50
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(s)
            for _ in range(n):
                B.llama_q8_attention(q, kc, vc, T, pos, nh, nkv, hd, stride, o, None, 0, s.cuda_stream)
            e1.record(s)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1000 / n
            visible = sum(pos + i + 1 for i in range(T))
            flops = 4.0 * nh * hd * visible
            tf = flops / (us * 1e-6) / 1e12
            out.append({"heads": f"{nh}/{nkv}x{hd}", "T": T, "index_pos": pos, "us": us, "tflops": tf,
                        "frac_fp32": tf / FP32_FMA_TFLOPS})
        del kc, vc
        torch.cuda.empty_cache()
    return out


def decode_timeline(model, cfg, n_steps, peak):
    """Per-family timeline of the decode step from the instrumented copy of
    the CUDA graph (llama_q8_profile_decode): exclusive time per launch (the
    step's time spent on it: from its dependency wait returning to the next
    launch's), span, algorithmic bytes, GB/s over both."""
    prof = model.profile_decode(n_steps)
    total_ms = sum(v[1] for v in prof.values())
    fams = {}
    for name, (n, ms, span_ms, nbytes) in prof.items():
        if n == 0:
            continue
        fams[name] = {"launches": n, "us_per_launch": 1000 * ms / n, "span_us_per_launch": 1000 * span_ms / n,
                      "bytes_per_launch": nbytes / n, "gbs": nbytes / (ms * 1e-3) / 1e9,
                      "gbs_over_span": nbytes / (span_ms * 1e-3) / 1e9, "share": ms / total_ms,
                      "us_per_token": 1000 * ms / n_steps}
    return fams, 1000 * total_ms / n_steps


def lm_head_variants(torch, B, synth, device, peak, prompt, n_steps):
    """The lm_head + argmax GEMV in the decode graph, row-parallel (persistent
    CTAs over 32-row tiles) against split-K (each tile's 576-wide range over a
    2-CTA cluster): its in-graph exclusive time from the timeline."""
    res = {}
    for name, splits in (("row_parallel", 0), ("split_k2", 2)):
        cfg, model = gpu_model(torch, B, synth, device, head_splits=splits)
        model.forward_argmax(prompt, 0)
        fams, step_us = decode_timeline(model, cfg, n_steps, peak)
        h = fams["gemv_head_argmax"]
        res[name] = {"us_per_launch": h["us_per_launch"], "gbs": h["gbs"], "frac": h["gbs"] / peak,
                     "step_us": step_us}
        model.close()
        torch.cuda.empty_cache()
    res["kept"] = min(("row_parallel", "split_k2"), key=lambda k: res[k]["us_per_launch"])
    return res


def attention_microbench(torch, B, synth, device, peak):
    """GQA decode attention at the 135M shape (9/3 heads of 64) and the 7B
    shape (32/8 heads of 128), kv_len 32..4096, the decode step's kernel
    (llama_q8_attention_decode). 100 launches, each on its own cache copy so
    that the K/V rows stream from HBM (one 4096-position cache is 6.3 / 33.6
    MB), are captured in a CUDA graph and replayed: the per-launch time is the
    kernel plus the graph's launch-to-launch gap, without host overhead."""
    out = []
    for nh, nkv, hd in ((9, 3, 64), (32, 8, 128)):
        stride = 4096
        ncopy = 8 if hd == 64 else 4
        kc = [torch.randn(nkv * stride * hd, device=device) for _ in range(ncopy)]
        vc = [torch.randn(nkv * stride * hd, device=device) for _ in range(ncopy)]
        q = torch.randn(nh * hd, device=device)
        o = torch.empty(nh * hd, device=device)
        for kv in (32, 256, 1024, 4096):
            s = torch.cuda.current_stream()
            for i in range(8):
                B.llama_q8_attention_decode(q, kc[i % ncopy], vc[i % ncopy], kv, nh, nkv, hd, stride, o,
                                            s.cuda_stream)
            torch.cuda.synchronize()
            n = 100
            g = torch.cuda.CUDAGraph()
            cs = torch.cuda.Stream()
            with torch.cuda.graph(g, stream=cs):
                for i in range(n):
                    B.llama_q8_attention_decode(q, kc[i % ncopy], vc[i % ncopy], kv, nh, nkv, hd, stride, o,
                                                cs.cuda_stream)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s = torch.cuda.current_stream()
            e0.record(s)
            g.replay()
            e1.record(s)
            torch.cuda.synchronize()
            del g
            us = e0.elapsed_time(e1) * 1000 / n
            algo = 2 * nkv * kv * hd * 4 + 2 * nh * hd * 4
            out.append({"heads": f"{nh}/{nkv}x{hd}", "kv_len": kv, "us": us, "gbs": algo / (us * 1e-6) / 1e9,
                        "frac": algo / (us * 1e-6) / 1e9 / peak})
        del kc, vc
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        dist_init(world, "nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from q8_quantized_llama_gb300 import binding as B
    from q8_quantized_llama_gb300 import synth
    B.lib()
    peak, peak_kind = hbm_peak()
    cfg, model = gpu_model(torch, B, synth, device)
    prompt = synth.prompt_ids(PROMPT_LEN, cfg["n_vocab"], SEED)
    d_prompt = torch.from_numpy(prompt).to(device)
    d_next = torch.zeros(1, dtype=torch.int32, device=device)
    d_out = torch.zeros(DECODE_STEPS, dtype=torch.int32, device=device)
    stream = torch.cuda.ExternalStream(model.stream(), device=device)

    def one_step():
        model.prefill_async(d_prompt, PROMPT_LEN, 0, d_next)
        model.decode_async(DECODE_STEPS, d_out)

    for _ in range(max(1, args.warmup)):
        one_step()
    model.sync()
    ref_tokens = np.concatenate([d_next.cpu().numpy(), d_out.cpu().numpy()])

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    launches0 = model.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        torch.cuda.nvtx.range_push("timed_region")
        for i in range(args.steps):
            ev[i][0].record(stream)
            model.prefill_async(d_prompt, PROMPT_LEN, 0, d_next)
            ev[i][1].record(stream)
            model.decode_async(DECODE_STEPS, d_out)
            ev[i][2].record(stream)
        model.sync()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
    barrier(world)
    gpu_launches = model.launch_count() - launches0
    pre_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[1].elapsed_time(e[2]) for e in ev]
    total_ms = sum(pre_ms) + sum(dec_ms)
    tokens = np.concatenate([d_next.cpu().numpy(), d_out.cpu().numpy()])
    assert np.array_equal(tokens, ref_tokens), "decode tokens changed between repetitions"
    value, t_max = aggregate_throughput(DECODE_STEPS * args.steps, sum(dec_ms) / 1000, world, device)
    clk = clocks.summary()
    if args.only == "decode":  # the timed region alone (launch-list captures)
        if rank == 0:
            print(json.dumps({"decode_ms_per_token": sum(dec_ms) / (DECODE_STEPS * args.steps),
                              "prefill_ms": statistics.median(pre_ms), "gpu_launches": gpu_launches}))
        model.close()
        return

    # end to end through the host API: the pages' loop, one synchronous call per token
    e2e_dec = []
    for i in range(args.warmup + args.steps):
        nxt = model.forward_argmax(prompt, 0)
        t0 = time.perf_counter()
        pos = PROMPT_LEN
        for _ in range(DECODE_STEPS):
            nxt = model.forward_argmax([nxt], pos)
            pos += 1
        if i >= args.warmup:
            e2e_dec.append(time.perf_counter() - t0)
    e2e_value, _ = aggregate_throughput(DECODE_STEPS * args.steps, sum(e2e_dec), world, device)

    # the decode step's timeline: the instrumented copy of the same CUDA graph (PDL chaining intact)
    model.forward_argmax(prompt, 0)
    fams, prof_step_us = decode_timeline(model, cfg, DECODE_STEPS, peak)
    dom_name = max(fams, key=lambda k: fams[k]["share"])
    dom = fams[dom_name]
    weights_bytes, kv_bytes = decode_bytes(cfg, PROMPT_LEN + (DECODE_STEPS + 1) / 2)
    traffic = NCU_TRAFFIC.get(dom_name)
    mean_kv = PROMPT_LEN + (DECODE_STEPS + 1) / 2
    traffic_bytes = None
    if traffic:  # scaled from the captured kv_len to the timed steps' mean, as the algorithmic bytes are
        traffic_bytes = traffic["bytes"] + traffic["kv_bytes_per_pos"] * (mean_kv - traffic["kv_len"])

    out = None
    if rank == 0:
        lm_head = lm_head_variants(torch, B, synth, device, peak, prompt, DECODE_STEPS)
        gemv7 = gemv_7b_roofline(torch, B, synth, device, peak)
        fmt_gemv = block_format_gemv_bench(torch, B, synth, device, peak)
        attn = attention_microbench(torch, B, synth, device, peak)
        attn_pf = attention_prefill_bench(torch, B, synth, device)
        sweep = linear_sweep(torch, B, synth, device, peak)
        gemm = gemm_microbench(torch, B, synth, device)
        model7 = decode_7b(torch, B, synth, device, peak)
        dec_tok_ms = [d / DECODE_STEPS for d in dec_ms]
        out = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": value / (1000.0 / PAGES_DECODE_MS),
            "vs_baseline_ref": "pages' M2 Max CPU Q8_0 decode, 7.40 ms/token (context only)",
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": "135M-shaped Q8_0 Llama (30x576, 9/3 heads, FFN 1536, vocab 49152, seed 0): "
                                   "203-token random prompt prefill + 128 greedy decode steps, fresh KV cache",
                       "prompt": PROMPT_LEN, "decode_steps": DECODE_STEPS,
                       "l2": "inputs larger than L2: each decode step streams 142.9 MB of Q8_0 weights"},
            "decode_ms_per_token": {"min": min(dec_tok_ms), "median": statistics.median(dec_tok_ms)},
            "prefill_ms": {"min": min(pre_ms), "median": statistics.median(pre_ms)},
            "prefill_tok_s": PROMPT_LEN * args.steps / (sum(pre_ms) / 1000),
            "clocks": clk,
            "e2e": {"value": e2e_value, "unit": "tokens/s",
                    "path": "llama_q8_forward_argmax per token (host ids in, host token out, one sync per token)",
                    "h2d_bytes_per_step": 4 * (PROMPT_LEN + DECODE_STEPS),
                    "d2h_bytes_per_step": 16 * (1 + DECODE_STEPS)},
            "gpu_launches": gpu_launches,
            "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": dom["gbs"], "peak": peak, "unit": "GB/s",
                         "frac": dom["gbs"] / peak, "peak_source": f"{peak_kind} HBM copy bandwidth (burst)",
                         "traffic": traffic_bytes,
                         "traffic_source": (f"ncu dram__bytes_read.sum + dram__bytes_write.sum of the same kernel "
                                            f"at kv_len {traffic['kv_len']}, scaled by {traffic['kv_bytes_per_pos']} "
                                            f"B per position to the mean kv_len {mean_kv}") if traffic else None,
                         "algorithmic_bytes_per_launch": dom["bytes_per_launch"],
                         "duration_us": dom["us_per_launch"], "span_us": dom["span_us_per_launch"],
                         "share_of_step": dom["share"],
                         "timing": "the decode graph's instrumented copy (same kernels and PDL chaining; each "
                                   "launch stamps %globaltimer at entry and when its dependency wait returns); "
                                   "duration = exclusive time per launch, averaged over 128 steps x 30 layers",
                         "note": "latency-bound: the kernel is a chain of dependent phases (norm, Q/K/V rows, "
                                 "row exchange, attention, partial exchange, W_o) for ~1.4 MB of bytes"},
            "decode_step_roofline": {"weights_bytes": weights_bytes, "kv_bytes_mean": kv_bytes,
                                     "roofline_us": (weights_bytes + kv_bytes) / (peak * 1e9) * 1e6,
                                     "graph_step_us": 1000 * statistics.median(dec_tok_ms),
                                     "instrumented_step_us": prof_step_us,
                                     "frac": ((weights_bytes + kv_bytes) / (peak * 1e9) * 1e6)
                                     / (1000 * statistics.median(dec_tok_ms))},
            "kernels": fams,
            "lm_head": lm_head,
            "gemv_7b": gemv7,
            "block_format_gemv": fmt_gemv,
            "attention_decode": attn,
            "attention_prefill": attn_pf,
            "linear_sweep": sweep,
            "gemm_prefill": gemm,
            "decode_7b": model7,
        }
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = run_cpu_baseline(args.cpu_baseline_seconds)
            # the same oracle on one thread, and on the two other configurations
            out["cpu_baseline_legs"] = {
                "c1_single_thread": run_cpu_baseline(max(15.0, args.cpu_baseline_seconds), threads=1),
                "c0": run_cpu_baseline(args.cpu_baseline_seconds, config="c0"),
                "c4": run_cpu_baseline(600.0, config="c4", timeout=900.0),
            }
    model.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out))


def main():
    args = parse_args()
    if args.cpu_baseline_worker:
        cpu_baseline_worker(args.cpu_baseline_seconds, args.cpu_baseline_threads, args.cpu_baseline_config)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.only == "decode7b":
        import torch
        torch.cuda.set_device(0)
        from q8_quantized_llama_gb300 import binding as B
        from q8_quantized_llama_gb300 import synth
        B.lib()
        print(json.dumps(decode_7b(torch, B, synth, torch.device("cuda", 0), hbm_peak()[0])))
        return
    if args.only in ("prefill", "prefill7b"):
        import torch
        torch.cuda.set_device(0)
        from q8_quantized_llama_gb300 import binding as B
        from q8_quantized_llama_gb300 import synth
        B.lib()
        print(json.dumps(prefill_only(torch, B, synth, torch.device("cuda", 0), args, args.only == "prefill7b")))
        return
    if args.only in ("sweep", "attnprefill"):
        import torch
        torch.cuda.set_device(0)
        from q8_quantized_llama_gb300 import binding as B
        from q8_quantized_llama_gb300 import synth
        B.lib()
        dev = torch.device("cuda", 0)
        if args.only == "sweep":
            print(json.dumps({"linear_sweep": linear_sweep(torch, B, synth, dev, hbm_peak()[0])}))
        else:
            print(json.dumps({"attention_prefill": attention_prefill_bench(torch, B, synth, dev)}))
        return
    if args.only == "profile":
        import torch
        torch.cuda.set_device(0)
        from q8_quantized_llama_gb300 import binding as B
        from q8_quantized_llama_gb300 import synth
        B.lib()
        dev = torch.device("cuda", 0)
        cfg, model = gpu_model(torch, B, synth, dev)
        prompt = synth.prompt_ids(PROMPT_LEN, cfg["n_vocab"], SEED)
        model.forward_argmax(prompt, 0)
        fams, step_us = decode_timeline(model, cfg, DECODE_STEPS, hbm_peak()[0])
        print(json.dumps({"instrumented_step_us": step_us, "kernels": fams,
                          "lm_head": lm_head_variants(torch, B, synth, dev, hbm_peak()[0], prompt, DECODE_STEPS)}))
        model.close()
        return
    if args.only == "gemm":
        import torch
        torch.cuda.set_device(0)
        from q8_quantized_llama_gb300 import binding as B
        from q8_quantized_llama_gb300 import synth
        B.lib()
        print(json.dumps({"gemm": gemm_microbench(torch, B, synth, torch.device("cuda", 0))}))
        return
    if args.only == "attn":
        import torch
        torch.cuda.set_device(0)
        from q8_quantized_llama_gb300 import binding as B
        from q8_quantized_llama_gb300 import synth
        B.lib()
        print(json.dumps({"attention_decode": attention_microbench(torch, B, synth, torch.device("cuda", 0),
                                                                    hbm_peak()[0])}))
        return
    if args.only in ("gemv7b", "formats"):
        import torch
        torch.cuda.set_device(0)
        from q8_quantized_llama_gb300 import binding as B
        from q8_quantized_llama_gb300 import synth
        B.lib()
        fn = gemv_7b_roofline if args.only == "gemv7b" else block_format_gemv_bench
        print(json.dumps(fn(torch, B, synth, torch.device("cuda", 0), hbm_peak()[0])))
        return
    run_ours(args)


if __name__ == "__main__":
    main()
