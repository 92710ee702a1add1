"""Benchmark: Flint NVFP4 MoE feed-forward + lm_head decode on one or more B300s.

Workload (default): the per-token FFN weight stream of Flint-40B-A2B -- 47 chained
MoE layers (hidden 2048, 256 experts of width 512, top-6 softmax-renormalised routing
with a Zipf(1.1) per-expert router bias, shared expert 1024, independent seeded
weights, RMSNorm eps 1e-6 between layers) followed by the 150,144-entry NVFP4 head,
batch-1 decode of 256 tokens.  One step = those 256 tokens, one after another.
Weights (21.5 GB NVFP4) are far larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl flint|reference]

Prints ONE JSON line (rank 0).  Under torchrun each rank decodes its own token
stream (replicas, weak scaling, no collective on the data path).
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
sys.path.insert(0, ROOT)

METRIC = "decode tok/s (MoE FFN+lm_head bytes) & % HBM roofline; prefill tok/s & % FP4 peak"
N_LAYERS = 47
N_TOKENS = 256
EPS = 1e-6
SEED = 0
ZIPF = 1.1
PREFILL_TOKENS = 4096


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"), "src": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "src": "fallback"}


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def slowest_rank_ms(ms: float, world: int, device) -> float:
    """The timed region's length on the slowest rank (ms): with world > 1 a MAX
    all-reduce over the ranks (any backend), then a barrier."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def whole_job_rate(world: int, steps: int, tokens_per_step: int, ms: float) -> float:
    """Tokens per second of the whole job: every rank decodes its own stream of
    tokens_per_step tokens per step, timed by the slowest rank's `ms`."""
    return world * steps * tokens_per_step / (ms / 1e3)


# ------------------------------------------------------------------------------ flint arm
def run_flint(args):
    import torch
    import torch.distributed as dist

    from sparse_moe_decode_02_b300 import flint, synth, workload

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    flint.lib()
    shape = synth.FLINT
    H = shape.hidden
    layers = [workload.build_layer(synth.LayerSpec(shape, seed=SEED, layer=l, zipf=ZIPF), dev)
              for l in range(args.layers)]
    head = workload.build_head(SEED, shape.vocab, H, dev)
    torch.cuda.synchronize()
    T = args.tokens
    x_tok = synth.tokens_bf16(SEED, H, T, stream=1 + rank, device=dev)
    argmax = torch.zeros(T, dtype=torch.int32, device=dev)
    ws = torch.empty(flint.workspace_bytes(flint.OP_MOE_DECODE, H, shape.n_experts, shape.top_k,
                                           shape.expert_width, shape.shared_width, 0, T),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        """256 tokens x 47 layers + head: one persistent kernel launch (public C ABI)."""
        flint.decode_tokens(layers, x_tok, head=head, rms_eps=EPS, argmax=argmax, ws=ws,
                            stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert flint.last_device_status() == 0, "device status after warm-up"
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ev[0].record(stream)
        for i in range(args.steps):
            step()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
    per_launch = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    ms = ev[0].elapsed_time(ev[-1])
    ms = slowest_rank_ms(ms, world, dev)
    tok_per_s = whole_job_rate(world, args.steps, T, ms)
    status = flint.last_device_status()

    layer_bytes = workload.layer_bytes_per_token(shape)
    head_b = workload.head_bytes(shape.vocab, H)
    token_bytes = args.layers * layer_bytes + head_b
    launch_bytes = T * token_bytes
    launch_ms = statistics.mean(per_launch)
    achieved = launch_bytes / (launch_ms * 1e-3) / 1e9
    peaks = _peaks()

    # end to end through the public API: host (pinned) inputs in, argmax out, per step
    x_host = x_tok.cpu().pin_memory()
    am_host = torch.empty(T, dtype=torch.int32).pin_memory()
    torch.cuda.synchronize()
    e2e_steps = max(1, min(args.steps, 3))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        x_tok.copy_(x_host, non_blocking=True)
        step()
        am_host.copy_(argmax, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_tok_s = world * e2e_steps * T / e2e_s

    result = {
        "metric": METRIC,
        "value": round(tok_per_s, 1),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4 weights (e2m1 + e4m3/16 + fp32), bf16 activations, fp32 accumulate",
        "data": "synthetic (seeded counter-based N(0,0.02) weights, N(0,1) bf16 tokens)",
        "config": {
            "workload": "Flint FFN weight stream: 47 MoE layers (H=2048, E=256 top-6 + "
                        "Zipf(1.1) bias, F=512, shared 1024) + NVFP4 lm_head V=150144, "
                        "B=1 decode of %d tokens per step" % T,
            "layers": args.layers, "tokens_per_step": T, "batch": 1,
            "bytes_per_token": token_bytes,
            "l2_policy": "inputs larger than L2 (21.5 GB of weights per token pass)",
            "parallelism": "replicas x%d" % world,
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "k_decode_persistent (flint_decode_tokens: %d tokens x %d layers + head)"
                      % (T, args.layers),
            "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"],
            "peak_src": peaks["src"],
            "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": None,
            "algorithmic_bytes_per_launch": launch_bytes,
            "algorithmic_bytes_per_token": token_bytes,
            "launch_ms": round(launch_ms, 4),
            "us_per_token": round(launch_ms * 1e3 / T, 3),
            "frac_of_8TBps": round(achieved / 8000.0, 4),
        },
        "e2e": {"value": round(e2e_tok_s, 1), "unit": "tok/s",
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * 4},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "device_status": status,
        "prefill": None,
        "sampling": measure_sampling(dev),
    }
    if not args.no_prefill:
        del layers, head
        torch.cuda.empty_cache()
        result["prefill"] = measure_prefill(dev)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args)
    if world > 1:
        dist.destroy_process_group()
    return result if rank == 0 else None


def measure_sampling(dev, reps: int = 20):
    """flint_sample_logits on fp32 logits over the Flint vocabulary (150,144) with the
    pages' settings (temperature 1.0, top-p 0.95, top-k 20), 1 and 8 rows; the logits
    are rewritten before each timed call, and the bytes counted are one read of them."""
    import torch

    from sparse_moe_decode_02_b300 import flint

    V = 150144
    res = {"workload": "sampling over V=150144 fp32 logits, T=1.0, top-p 0.95, top-k 20"}
    for B in (1, 8):
        g = torch.Generator(device=dev).manual_seed(SEED + B)
        lg = torch.randn(B, V, device=dev, generator=g) * 3
        u = torch.rand(B, device=dev, generator=g)
        for _ in range(3):
            flint.sample_logits(lg, u)
        ts = []
        for _ in range(reps):
            lg.mul_(1.0)                       # logits rewritten: a new head output
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            flint.sample_logits(lg, u)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = sum(ts) / len(ts)
        res["B%d_us" % B] = round(ms * 1e3, 2)
        res["B%d_read_GBs" % B] = round(B * V * 4 / (ms * 1e-3) / 1e9, 1)
    return res


def measure_prefill(dev, reps: int = 10):
    """Prompt processing on one Flint layer: 4096 tokens, Zipf(1.1) router bias."""
    import torch

    from sparse_moe_decode_02_b300 import flint, synth, workload

    shape = synth.FLINT
    T = PREFILL_TOKENS
    layer = workload.build_layer(synth.LayerSpec(shape, seed=SEED, layer=0, zipf=ZIPF), dev)
    x = synth.tokens_bf16(SEED, shape.hidden, T, stream=11, device=dev)
    out = torch.empty(T, shape.hidden, dtype=torch.float32, device=dev)
    idx = torch.empty(T, shape.top_k, dtype=torch.int32, device=dev)
    counts = torch.empty(shape.n_experts, dtype=torch.int32, device=dev)
    ws = torch.empty(flint.workspace_bytes(flint.OP_MOE_PREFILL, shape.hidden, shape.n_experts,
                                           shape.top_k, shape.expert_width, shape.shared_width, 0,
                                           T), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    # a buffer larger than L2, rewritten between timed runs
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for _ in range(3):
        flint.moe_prefill(layer, x, out=out, expert_counts=counts, topk_idx=idx, ws=ws)
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        flint.moe_prefill(layer, x, out=out, expert_counts=counts, topk_idx=idx, ws=ws)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    cnt = counts.cpu().numpy()
    H, F, Fs, k = shape.hidden, shape.expert_width, shape.shared_width, shape.top_k
    flops = 2.0 * T * k * 3 * H * F + 2.0 * T * 3 * H * Fs          # FP4 products
    router_flops = 2.0 * T * shape.n_experts * H
    nv = lambda n: n // 2 + n // 16
    touched = int((cnt > 0).sum())
    weight_bytes = touched * 3 * nv(H * F) + 3 * nv(H * Fs) + shape.n_experts * H * 2
    bytes_ = weight_bytes + T * H * 2 + T * H * 4
    peaks = _peaks()
    fp4_peak = peaks["bf16_tflops"] * 6.0                              # nominal fp4/bf16 = 6
    tflops = flops / (ms * 1e-3) / 1e12
    del layer, ws, flush
    return {
        "workload": "Flint prompt processing: one MoE layer, %d tokens, Zipf(1.1) bias" % T,
        "value": round(T / (ms * 1e-3), 1), "unit": "tok/s", "ms": round(ms, 4),
        "fp4_gflop": round(flops / 1e9, 1), "router_gflop": round(router_flops / 1e9, 2),
        "tflops": round(tflops, 1), "fp4_peak_tflops": round(fp4_peak, 1),
        "fp4_peak_src": "measured bf16 %s x 6 (nominal FP4/BF16 dense ratio)" % peaks["src"],
        "frac_fp4_peak": round(tflops / fp4_peak, 4),
        "experts_touched": touched, "bytes": bytes_,
        "frac_hbm": round(bytes_ / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
        "l2_policy": "256 MB buffer rewritten before each timed run",
    }


# ------------------------------------------------------------------------------ oracle arm
def oracle_decode_sample(n_tokens: int, n_layers: int):
    """Times the CPU oracle on `n_tokens` tokens (processed together: the oracle threads
    over tokens) through the first `n_layers` chained layers and the head.  Returns
    (seconds of oracle compute per token through all 47 layers + head, threads used,
    description).  Weight generation is excluded from the timing."""
    import numpy as np

    import oracle
    from sparse_moe_decode_02_b300 import synth

    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from helpers import bits16, oracle_layer, oracle_routes

    shape = synth.FLINT
    H = shape.hidden
    threads = min(oracle.get_threads(), n_tokens)
    xb = bits16(synth.tokens_bf16(SEED, H, n_tokens, stream=1))
    hres = None
    layer_s = 0.0
    for l in range(n_layers):
        spec = synth.LayerSpec(shape, seed=SEED, layer=l, zipf=ZIPF)
        _, idx, _ = oracle_routes(oracle, spec, xb)
        L = oracle_layer(oracle, spec, experts=np.unique(idx))
        t0 = time.perf_counter()
        out, _, _ = oracle.moe_forward(L, xb, residual=hres)
        xb = np.stack([oracle.rmsnorm_bf16(out[t], EPS) for t in range(n_tokens)])
        layer_s += time.perf_counter() - t0
        hres = out
    hq, _ = oracle.quantize_nvfp4(synth.head_bf16(SEED, shape.vocab, H))
    t0 = time.perf_counter()
    oracle.lm_head(hq, xb)
    head_s = time.perf_counter() - t0
    per_token = (layer_s / n_layers * N_LAYERS + head_s) / n_tokens
    desc = ("%d tokens together x the first %d of 47 layers (oracle-selected experts), then "
            "the full 150144-row head; per-token time = (mean layer time x 47 + head time) / "
            "%d" % (n_tokens, n_layers, n_tokens))
    return per_token, threads, desc


def cpu_baseline(args):
    per_tok, threads, desc = oracle_decode_sample(args.cpu_tokens, args.cpu_layers)
    return {"value": round(1.0 / per_tok, 4), "unit": "tok/s", "cores": threads,
            "kind": "oracle", "sample": desc}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return None
    times = []
    threads, desc = None, None
    for _ in range(args.warmup + args.steps):
        per_tok, threads, desc = oracle_decode_sample(args.cpu_tokens, args.cpu_layers)
        times.append(per_tok)
    timed = times[args.warmup:]
    tok_s = 1.0 / statistics.mean(timed)
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(tok_s, 4),
        "unit": "tok/s",
        "n_gpus": 0,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(statistics.mean(timed) * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp64 (CPU oracle)",
        "data": "synthetic (seeded, same generator as the flint arm)",
        "config": {"workload": "Flint FFN weight stream (47 layers + NVFP4 head), B=1 decode; "
                               "each step is a bounded sample, see cpu_baseline.sample"},
        "cpu_baseline": {"value": round(tok_s, 4), "unit": "tok/s", "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(tok_s, 4), "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="flint", choices=["flint", "reference"])
    ap.add_argument("--tokens", type=int, default=N_TOKENS)
    ap.add_argument("--layers", type=int, default=N_LAYERS)
    ap.add_argument("--cpu-layers", type=int, default=2)
    ap.add_argument("--cpu-tokens", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the prompt-processing layer (prints its object)")
    args = ap.parse_args()
    if args.prefill_only and args.impl == "flint":
        import torch
        torch.cuda.set_device(0)
        from sparse_moe_decode_02_b300 import flint
        flint.lib()
        print(json.dumps(measure_prefill(torch.device("cuda", 0), reps=args.steps)), flush=True)
        return
    res = run_reference(args) if args.impl == "reference" else run_flint(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
