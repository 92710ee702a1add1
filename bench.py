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


NOMINAL_FP4_TFLOPS = 13500.0     # dense NVFP4 per GPU, NVIDIA's figure (without 2:4 sparsity)


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"), "src": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "src": "fallback"}


def _sha1(path):
    import hashlib
    return hashlib.sha1(open(path, "rb").read()).hexdigest()


def decode_traffic(tokens: int, layers: int):
    """DRAM bytes (read + write) of one decode launch from the committed ncu capture
    (profiles/k_decode_dram.md: a smaller launch of the same kernel, scaled by the
    token-layers and head passes it processes), or None when the kernel source changed
    since the capture."""
    p = os.path.join(ROOT, "profiles", "k_decode_dram.md")
    if not os.path.exists(p):
        return None
    fields = {}
    for ln in open(p):
        if ln.startswith("- ") and ":" in ln:
            k, v = ln[2:].split(":", 1)
            fields[k.strip()] = v.strip().split()[0]
    src = os.path.join(ROOT, "sparse_moe_decode_02_b300", "csrc", "decode.cu")
    if fields.get("decode.cu sha1") != _sha1(src):
        return None
    try:
        per_tl = float(fields["dram bytes per token-layer"])
        per_head = float(fields["dram bytes per head pass"])
    except (KeyError, ValueError):
        return None
    return tokens * (layers * per_tl + per_head)


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
            "kernel": "k_decode<2> (flint_decode_tokens: %d tokens x %d layers + head)"
                      % (T, args.layers),
            "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"],
            "peak_src": peaks["src"],
            "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": decode_traffic(T, args.layers),
            "traffic_src": "profiles/k_decode_dram.md (ncu dram__bytes_read.sum + "
                           "dram__bytes_write.sum of a smaller launch, scaled per token-layer "
                           "and head pass; null if decode.cu changed since)",
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
    }
    if not args.decode_only:
        result["sampling"] = measure_sampling(dev)
        # the same step with the token drawn in the launch (top-k 20, top-p 0.95, T = 1)
        u = torch.rand(T, device=dev, generator=torch.Generator(device=dev).manual_seed(SEED))
        toks = torch.empty(T, dtype=torch.int32, device=dev)
        fused = lambda: flint.decode_tokens_sample(layers, x_tok, head, u, tokens=toks, rms_eps=EPS,
                                                   ws=ws, stream=stream)
        fused()
        torch.cuda.synchronize()
        ms_f = _time_ms(fused, 2, stream)
        result["sampling"]["fused_decode"] = {
            "value": round(T / (ms_f * 1e-3), 1), "unit": "tok/s", "ms_per_step": round(ms_f, 3),
            "workload": "the decode step with each token drawn inside the launch "
                        "(flint_decode_tokens_sample: top-k 20, top-p 0.95, temperature 1)"}
        result["config3_lm_head"] = measure_lm_head(dev, head)
    del layers, head
    torch.cuda.empty_cache()
    if not args.decode_only:
        result["config2_layer"] = measure_layer(dev)
        result["dense_layers"] = measure_dense(dev)
        fp4 = measure_fp4_peak(dev)
        result["fp4_peak"] = fp4
        if not args.no_prefill:
            result["prefill"] = measure_prefill(dev, fp4_tflops=fp4["tflops"])
    if rank == 0 and not args.no_cpu_baseline and not args.decode_only:
        result["cpu_baseline"] = cpu_baseline(args)
    if world > 1:
        dist.destroy_process_group()
    return result if rank == 0 else None


def _time_ms(fn, reps, stream=None, inner=1):
    """Median ms of one `fn` call over `reps` timed runs of `inner` back-to-back calls
    (CUDA events on the current stream)."""
    import torch
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(inner):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / inner)
    return statistics.median(times)


def measure_lm_head(dev, head, reps: int = 10):
    """The standalone NVFP4 lm_head (flint_lm_head): 150,144 x 2048 weights, batch 1 and
    batch 8, fp32 logits plus argmax; ten calls back to back per timed run.  The 173 MB of
    weights exceed L2, so every call streams them from HBM."""
    import torch

    from sparse_moe_decode_02_b300 import flint, synth, workload

    shape = synth.FLINT
    H, V = shape.hidden, shape.vocab
    peaks = _peaks()
    wbytes = workload.head_bytes(V, H)
    res = {"workload": "NVFP4 lm_head %d x %d, fp32 logits + argmax" % (V, H)}
    for B in (1, 8):
        x = synth.tokens_bf16(SEED, H, B, stream=21, device=dev)
        lg = torch.empty(B, V, dtype=torch.float32, device=dev)
        am = torch.empty(B, dtype=torch.int32, device=dev)
        for _ in range(3):
            flint.lm_head(head, x, logits=lg, argmax=am)
        torch.cuda.synchronize()
        ws = torch.empty(flint.workspace_bytes(flint.OP_LM_HEAD, H, 0, 0, 0, 0, V, B),
                         dtype=torch.uint8, device=dev)
        ms = _time_ms(lambda: flint.lm_head(head, x, logits=lg, argmax=am, ws=ws), reps, inner=10)
        moved = wbytes + B * (H * 2 + V * 4 + 4)
        gbs = moved / (ms * 1e-3) / 1e9
        res["B%d" % B] = {"value": round(B / (ms * 1e-3), 1), "unit": "tok/s",
                          "us": round(ms * 1e3, 2), "bytes": moved, "GBs": round(gbs, 1),
                          "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}
    res["kernel"] = "k_lm_head (profiles/k_lm_head_dram.md)"
    return res


def measure_layer(dev, reps: int = 5):
    """One Flint MoE layer (no router bias), batch 1, 1000 seeded tokens one after another
    in one flint_decode_tokens launch: tokens/s and bytes per token (router 1 MB + 6
    routed experts + shared expert = 15,204,352 B)."""
    import torch

    from sparse_moe_decode_02_b300 import flint, synth, workload

    shape = synth.FLINT
    H, T = shape.hidden, 1000
    layer = workload.build_layer(synth.LayerSpec(shape, seed=SEED, layer=0), dev)
    x = synth.tokens_bf16(SEED, H, T, stream=2, device=dev)
    out = torch.empty(T, H, dtype=torch.float32, device=dev)
    for _ in range(2):
        flint.decode_tokens([layer], x, out=out)
    torch.cuda.synchronize()
    ms = _time_ms(lambda: flint.decode_tokens([layer], x, out=out), reps)
    per_tok = workload.layer_bytes_per_token(shape)
    gbs = per_tok * T / (ms * 1e-3) / 1e9
    peaks = _peaks()
    del layer
    return {"workload": "one Flint MoE layer (H=2048, E=256 top-6, F=512, shared 1024), "
                        "batch 1, %d tokens per launch" % T,
            "value": round(T / (ms * 1e-3), 1), "unit": "tok/s", "ms": round(ms, 4),
            "us_per_token": round(ms * 1e3 / T, 3), "bytes_per_token": per_tok,
            "GBs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "note": "consecutive tokens of one layer reuse experts already in L2 (453 MB of "
                    "routed weights, 126 MB L2): DRAM traffic is below the algorithmic bytes"}


def measure_dense(dev, reps: int = 3, T: int = 256):
    """The model's two dense SwiGLU layers (width 6,144, no router) decoded in one launch,
    batch 1, T tokens one after another: tokens/s and bytes per token."""
    import torch

    from sparse_moe_decode_02_b300 import flint, synth, workload

    shape = synth.FLINT_DENSE
    H = shape.hidden
    layers = [workload.build_layer(synth.LayerSpec(shape, seed=SEED, layer=100 + l), dev)
              for l in range(2)]
    x = synth.tokens_bf16(SEED, H, T, stream=12, device=dev)
    out = torch.empty(T, H, dtype=torch.float32, device=dev)
    for _ in range(2):
        flint.decode_tokens(layers, x, out=out)
    torch.cuda.synchronize()
    ms = _time_ms(lambda: flint.decode_tokens(layers, x, out=out), reps)
    per_tok = 2 * workload.layer_bytes_per_token(shape)
    gbs = per_tok * T / (ms * 1e-3) / 1e9
    peaks = _peaks()
    del layers
    return {"workload": "2 dense SwiGLU layers (H=2048, width 6144, no router), batch 1, "
                        "%d tokens per launch" % T,
            "value": round(T / (ms * 1e-3), 1), "unit": "tok/s", "ms": round(ms, 4),
            "us_per_token": round(ms * 1e3 / T, 3), "bytes_per_token": per_tok,
            "GBs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)}


def measure_fp4_peak(dev, iters: int = 20000):
    """Block-scaled FP4 tensor-core throughput (flint_bench_fp4_mma mode 0: M = 128,
    N = 128, K = 64 tcgen05.mma kind::mxf4nvf4 back to back, operands in shared memory
    and TMEM) on every SM, timed with CUDA events."""
    import torch

    from sparse_moe_decode_02_b300 import flint

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flint.bench_fp4_mma(0, 200, sms)
    torch.cuda.synchronize()
    ms = _time_ms(lambda: flint.bench_fp4_mma(0, iters, sms), 3)
    flop = sms * iters * 8 * 2.0 * 128 * 128 * 64
    return {"tflops": round(flop / (ms * 1e-3) / 1e12, 1), "ctas": sms, "iters": iters,
            "ms": round(ms, 3), "nominal_tflops": NOMINAL_FP4_TFLOPS,
            "shape": "tcgen05.mma kind::mxf4nvf4 block16, M=128 N=128 K=64, 8 per iteration"}


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


def measure_prefill(dev, reps: int = 10, fp4_tflops: float | None = None):
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
    # the larger of the measured tcgen05 FP4 peak and NVIDIA's dense figure
    fp4_peak = max(fp4_tflops or 0.0, NOMINAL_FP4_TFLOPS)
    tflops = flops / (ms * 1e-3) / 1e12
    del layer, ws, flush
    return {
        "workload": "Flint prompt processing: one MoE layer, %d tokens, Zipf(1.1) bias" % T,
        "value": round(T / (ms * 1e-3), 1), "unit": "tok/s", "ms": round(ms, 4),
        "fp4_gflop": round(flops / 1e9, 1), "router_gflop": round(router_flops / 1e9, 2),
        "tflops": round(tflops, 1), "fp4_peak_tflops": round(fp4_peak, 1),
        "fp4_peak_src": "max(measured tcgen05 mxf4nvf4 %s TF/s, NVIDIA dense %s TF/s)" % (
            fp4_tflops, NOMINAL_FP4_TFLOPS),
        "frac_fp4_peak": round(tflops / fp4_peak, 4),
        "experts_touched": touched, "bytes": bytes_,
        "frac_hbm": round(bytes_ / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
        "l2_policy": "256 MB buffer rewritten before each timed run",
    }


# ------------------------------------------------------------------------------ oracle arm
def _gen_device():
    """Where the seeded bf16 draws are made for the oracle (the same bits on any device;
    only the oracle's own arithmetic is timed)."""
    try:
        import torch
        return "cuda" if torch.cuda.is_available() else "cpu"
    except ImportError:
        return "cpu"


class OracleDecode:
    """The CPU oracle decoding `n_tokens` tokens (processed together: the oracle threads
    over tokens) through the 47 chained Flint layers and the 150,144-row head.  The
    weights each token's route needs are generated and quantised once (one untimed pass
    over the chain finds the routes); run() times the oracle's arithmetic only."""

    def __init__(self, n_tokens: int, n_layers: int = N_LAYERS):
        import numpy as np

        import oracle
        from oracle import seeded
        from sparse_moe_decode_02_b300 import synth

        self.np, self.oracle = np, oracle
        shape = synth.FLINT
        gen = _gen_device()
        self.n_tokens, self.n_layers = n_tokens, n_layers
        self.x = seeded.bits16(synth.tokens_bf16(SEED, shape.hidden, n_tokens, stream=1))
        self.layers = []
        xb, h = self.x, None
        for l in range(n_layers):
            spec = synth.LayerSpec(shape, seed=SEED, layer=l, zipf=ZIPF)
            _, idx, _ = seeded.routes(spec, xb)
            L = seeded.layer(spec, experts=np.unique(idx), gen_device=gen)
            h, _, _ = oracle.moe_forward(L, xb, residual=h)
            xb = np.stack([oracle.rmsnorm_bf16(h[t], EPS) for t in range(n_tokens)])
            self.layers.append(L)
        self.head = seeded.head(SEED, shape.vocab, shape.hidden, gen)
        self.threads = min(oracle.get_threads(), n_tokens)

    def run(self) -> float:
        """Seconds of oracle compute for the tokens through every layer and the head."""
        np, oracle = self.np, self.oracle
        t0 = time.perf_counter()
        xb, h = self.x, None
        for L in self.layers:
            h, _, _ = oracle.moe_forward(L, xb, residual=h)
            xb = np.stack([oracle.rmsnorm_bf16(h[t], EPS) for t in range(self.n_tokens)])
        oracle.lm_head(self.head, xb)
        return time.perf_counter() - t0

    def sample(self) -> str:
        return ("%d tokens (batched) x %d chained Flint layers (oracle-selected experts) + the "
                "150144-row head, fp64; weight generation and quantisation not timed"
                % (self.n_tokens, self.n_layers))


def oracle_units(dec: OracleDecode, n_tokens: int = 16):
    """CPU oracle rates of the other benchmarked configurations on bounded samples:
    config 2 (one Flint layer, no bias), config 3 (the head, batch 1 and 8; reuses the
    decode's head) and config 5 (the prompt layer with activation quantisation)."""
    import numpy as np

    import oracle
    from oracle import seeded
    from sparse_moe_decode_02_b300 import synth

    gen = _gen_device()
    shape = synth.FLINT
    H = shape.hidden
    res = {}
    x = seeded.bits16(synth.tokens_bf16(SEED, H, n_tokens, stream=2))
    spec = synth.LayerSpec(shape, seed=SEED, layer=0)
    _, idx, _ = seeded.routes(spec, x)
    L = seeded.layer(spec, experts=np.unique(idx), gen_device=gen)
    t0 = time.perf_counter()
    oracle.moe_forward(L, x)
    s2 = time.perf_counter() - t0
    res["config2_layer"] = {"value": round(n_tokens / s2, 3), "unit": "tok/s",
                            "sample": "%d tokens of one Flint layer" % n_tokens}
    for B in (1, 8):
        xb = seeded.bits16(synth.tokens_bf16(SEED, H, B, stream=21))
        t0 = time.perf_counter()
        oracle.lm_head(dec.head, xb)
        s3 = time.perf_counter() - t0
        res["config3_lm_head_B%d" % B] = {"value": round(B / s3, 3), "unit": "tok/s",
                                          "sample": "the full head, %d row(s) of x" % B}
    spec5 = synth.LayerSpec(shape, seed=SEED, layer=0, zipf=ZIPF)
    x5 = seeded.bits16(synth.tokens_bf16(SEED, H, n_tokens, stream=11))
    _, idx5, _ = seeded.routes(spec5, x5)
    L5 = seeded.layer(spec5, experts=np.unique(idx5), gen_device=gen)
    t0 = time.perf_counter()
    oracle.moe_forward(L5, x5, quantize_acts=True)
    s5 = time.perf_counter() - t0
    res["config5_prefill"] = {"value": round(n_tokens / s5, 3), "unit": "tok/s",
                              "sample": "%d of the 4096 prompt tokens (activations quantised "
                                        "to NVFP4 as the prompt path does)" % n_tokens}
    return res


def cpu_baseline(args):
    dec = OracleDecode(args.cpu_tokens)
    secs = dec.run()
    out = {"value": round(dec.n_tokens / secs, 4), "unit": "tok/s", "cores": dec.threads,
           "kind": "oracle", "sample": dec.sample(), "seconds": round(secs, 2)}
    out["units"] = oracle_units(dec)
    return out


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return None
    dec = OracleDecode(args.cpu_tokens)
    times = [dec.run() for _ in range(args.warmup + args.steps)]
    timed = times[args.warmup:]
    secs = statistics.mean(timed)
    tok_s = dec.n_tokens / secs
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(tok_s, 4),
        "unit": "tok/s",
        "n_gpus": 0,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp64 (CPU oracle)",
        "data": "synthetic (seeded, same generator as the flint arm)",
        "config": {"workload": "Flint FFN weight stream (47 layers + NVFP4 head), B=1 decode; "
                               "each step is a bounded sample, see cpu_baseline.sample"},
        "cpu_baseline": {"value": round(tok_s, 4), "unit": "tok/s", "cores": dec.threads,
                         "kind": "oracle", "sample": dec.sample()},
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
    ap.add_argument("--cpu-tokens", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--decode-only", action="store_true",
                    help="the decode line alone (no other measurements, no CPU baseline)")
    ap.add_argument("--case", default=None, choices=["prefill", "layer", "lm_head", "fp4", "dense"],
                    help="time one other configuration alone (prints its object)")
    ap.add_argument("--prefill-only", action="store_true", help="same as --case prefill")
    args = ap.parse_args()
    if args.prefill_only:
        args.case = "prefill"
    if args.case and args.impl == "flint":
        import torch
        torch.cuda.set_device(0)
        from sparse_moe_decode_02_b300 import flint, synth, workload
        flint.lib()
        dev = torch.device("cuda", 0)
        if args.case == "prefill":
            res = measure_prefill(dev, reps=args.steps)
        elif args.case == "layer":
            res = measure_layer(dev, reps=args.steps)
        elif args.case == "dense":
            res = measure_dense(dev, reps=args.steps)
        elif args.case == "lm_head":
            head = workload.build_head(SEED, synth.FLINT.vocab, synth.FLINT.hidden, dev)
            res = measure_lm_head(dev, head, reps=args.steps)
        else:
            res = measure_fp4_peak(dev)
        print(json.dumps(res), flush=True)
        return
    res = run_reference(args) if args.impl == "reference" else run_flint(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
