"""Oracle-side layers and heads built from the seeded workload generator.

TEST INFRASTRUCTURE, like the rest of this package (imported only by ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``).  The weights come from
the library's seeded input generator (``synth``: counter-based hashes and a normal
table, the same bits on any device, none of the method's arithmetic); everything the
method computes on them -- quantisation, routing, the experts, the head -- is the
oracle's own (``flint_oracle.c``).
"""
from __future__ import annotations

import numpy as np
import torch

from sparse_moe_decode_02_b300 import synth

from . import Layer, NVFP4, quantize_nvfp4, router


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> its uint16 bit patterns (numpy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def stack(spec: synth.LayerSpec, kind: int, experts, gen_device="cpu") -> NVFP4:
    """NVFP4 stack of one matrix kind, quantised by the oracle; only `experts` are
    generated (the other matrices are zero).  `gen_device` only sets where the bf16
    draws are made."""
    n, r, c = spec.dims(kind)
    codes = np.zeros((n, r, c // 2), np.uint8)
    scales = np.zeros((n, r, c // 16), np.uint8)
    tsc = np.ones(n, np.float32)
    ex = sorted(set(int(e) for e in experts))
    for i in range(0, len(ex), 16):                  # 16 matrices per quantiser call
        part = ex[i:i + 16]
        q, st = quantize_nvfp4(spec.weights_bf16(kind, device=gen_device, experts=part).cpu())
        assert st == 0
        codes[part], scales[part], tsc[part] = q.codes, q.scales, q.tsc
    return NVFP4(codes, scales, tsc)


def layer(spec: synth.LayerSpec, experts=None, gen_device="cpu") -> Layer:
    """Oracle layer from the same seeded bf16 tensors as the device layer."""
    s = spec.shape
    experts = range(s.n_experts) if experts is None else experts
    rw = bits16(spec.weights_bf16(synth.KIND_ROUTER, device=gen_device)[0])
    mk = lambda kind, ex: stack(spec, kind, ex, gen_device)
    return Layer(rw, spec.bias(), mk(synth.KIND_GATE, experts), mk(synth.KIND_UP, experts),
                 mk(synth.KIND_DOWN, experts), mk(synth.KIND_SH_GATE, [0]),
                 mk(synth.KIND_SH_UP, [0]), mk(synth.KIND_SH_DOWN, [0]), s.top_k,
                 router_score=spec.router_score)


def router_only_layer(spec: synth.LayerSpec) -> Layer:
    """A layer whose expert stacks are empty placeholders: enough for routing."""
    s = spec.shape
    z = lambda n, r, c: NVFP4(np.zeros((n, r, c // 2), np.uint8), np.zeros((n, r, c // 16), np.uint8),
                              np.ones(n, np.float32))
    H, F, Fs = s.hidden, s.expert_width, s.shared_width
    return Layer(bits16(spec.weights_bf16(synth.KIND_ROUTER)[0]), spec.bias(), z(1, F, H), z(1, F, H),
                 z(1, H, F), z(1, Fs, H), z(1, Fs, H), z(1, H, Fs), s.top_k,
                 router_score=spec.router_score)


def routes(spec: synth.LayerSpec, x_bits: np.ndarray):
    """(logits [T, E], idx [T, k], w [T, k]) from the oracle router."""
    L = router_only_layer(spec)
    out = [router(L, x_bits[t]) for t in range(x_bits.shape[0])]
    return (np.stack([o[0] for o in out]), np.stack([o[1] for o in out]),
            np.stack([o[2] for o in out]))


def head(seed: int, vocab: int, hidden: int, gen_device="cpu") -> NVFP4:
    """The output head [1, V, H], quantised by the oracle."""
    q, st = quantize_nvfp4(synth.head_bf16(seed, vocab, hidden, device=gen_device).cpu())
    assert st == 0
    return q
