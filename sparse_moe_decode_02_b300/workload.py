"""Device-side workloads: seeded synthetic Flint layers and heads, quantised to NVFP4 by
the library itself (flint_quantize_nvfp4), ready for flint_moe_decode / flint_lm_head /
flint_moe_prefill.  Shapes follow "Flint: 125 tokens a second is what 2.5B active
parameters buy at 273 GB/s", section "The shape, read from the headers".
"""
from __future__ import annotations

import torch

from . import flint, synth


def build_layer(spec: synth.LayerSpec, device="cuda", stream=None) -> flint.MoELayer:
    """Generate one layer's bf16 weights on the device and quantise them."""
    s = spec.shape

    def q(kind):
        w = spec.weights_bf16(kind, device=device)
        m = flint.quantize_nvfp4(w, stream=stream)
        del w
        return m

    router = spec.weights_bf16(synth.KIND_ROUTER, device=device)[0].contiguous()
    bias = spec.bias() if s.n_experts > 0 else None
    bias_t = None if bias is None else torch.from_numpy(bias).to(device)
    if s.n_experts == 0:
        # a dense layer: no routed stacks (empty placeholders; the library ignores them)
        empty = lambda: flint.NVFP4(torch.empty(0, 0, s.hidden // 2, dtype=torch.uint8, device=device),
                                    torch.empty(0, 0, s.hidden // 16, dtype=torch.uint8, device=device),
                                    torch.empty(0, dtype=torch.float32, device=device))
        gate, up, down = empty(), empty(), empty()
        sh_gate, sh_up, sh_down = q(synth.KIND_SH_GATE), q(synth.KIND_SH_UP), q(synth.KIND_SH_DOWN)
        return flint.MoELayer(router, None, gate, up, down, sh_gate, sh_up, sh_down, 0,
                              mma_scales=None, router_score=spec.router_score)
    gate, up, down = q(synth.KIND_GATE), q(synth.KIND_UP), q(synth.KIND_DOWN)
    sh_gate, sh_up, sh_down = q(synth.KIND_SH_GATE), q(synth.KIND_SH_UP), q(synth.KIND_SH_DOWN)
    stacks = (gate, up, down, sh_gate, sh_up, sh_down)
    # the prompt path's MMA scale copies exist for 128-row, 64-column multiples
    mma = None
    if all(m.shape[1] % 128 == 0 and m.shape[2] % 64 == 0 for m in stacks):
        mma = tuple(flint.nvfp4_mma_scales(m, stream=stream) for m in stacks)
    return flint.MoELayer(router, bias_t, gate, up, down, sh_gate, sh_up, sh_down, s.top_k,
                          mma_scales=mma, router_score=spec.router_score)


def build_head(seed: int, vocab: int, hidden: int, device="cuda", stream=None) -> flint.NVFP4:
    w = synth.head_bf16(seed, vocab, hidden, device=device)
    m = flint.quantize_nvfp4(w, stream=stream)
    del w
    return m


def layer_bytes_per_token(shape: synth.MoeShape) -> int:
    """Algorithmic weight bytes one decode token reads from one layer: the bf16 router,
    top_k routed experts and the shared expert (gate, up, down) in NVFP4 (0.5 B codes +
    1/16 B scales per weight).  A dense layer (no experts) reads its block only."""
    H, F, Fs, k, E = (shape.hidden, shape.expert_width, shape.shared_width, shape.top_k,
                      shape.n_experts)
    nv = lambda n: n // 2 + n // 16
    return E * H * 2 + k * 3 * nv(H * F) + 3 * nv(H * Fs)


def head_bytes(vocab: int, hidden: int) -> int:
    n = vocab * hidden
    return n // 2 + n // 16
