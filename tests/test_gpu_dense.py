"""Dense SwiGLU layers in the decode chain (the model's two dense MLP layers, width
6,144: "Flint: 125 tokens a second is what 2.5B active parameters buy at 273 GB/s",
section "Built from scratch?"): layers with no router and no routed experts, alone and
between MoE layers, checked layer by layer against the oracle (teacher-forced through
flint_decode_tokens_trace)."""
import numpy as np
import pytest
import torch

from helpers import assert_close, bits16, check_routing, oracle_layer, oracle_routes
from sparse_moe_decode_02_b300 import flint, synth, workload

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS = 1e-6
SMALL_DENSE = synth.MoeShape(hidden=256, n_experts=0, top_k=0, expert_width=0, shared_width=384,
                             vocab=4096)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flint.lib()


def _chain(orc, shapes, T, seed):
    specs = [synth.LayerSpec(s, seed=seed, layer=l, zipf=1.1 if s.n_experts else None)
             for l, s in enumerate(shapes)]
    layers = [workload.build_layer(s, DEV) for s in specs]
    H, L = shapes[0].hidden, len(shapes)
    kmax = max(s.top_k for s in shapes)
    x = synth.tokens_bf16(seed, H, T, stream=8)
    out = torch.empty(T, H, dtype=torch.float32, device=DEV)
    xt = torch.empty(T, L, H, dtype=torch.bfloat16, device=DEV)
    ht = torch.empty(T, L, H, dtype=torch.float32, device=DEV)
    tidx = torch.empty(T, L, max(kmax, 1), dtype=torch.int32, device=DEV)
    tw = torch.empty(T, L, max(kmax, 1), dtype=torch.float32, device=DEV)
    flint.decode_tokens(layers, x.to(DEV), rms_eps=EPS, out=out, topk_idx=tidx, topk_w=tw,
                        x_trace=xt, h_trace=ht)
    torch.cuda.synchronize()
    assert flint.last_device_status() == 0
    xt, ht = bits16(xt), ht.cpu().numpy().astype(np.float64)
    g_out = out.cpu().numpy().astype(np.float64)
    gi, gw = tidx.cpu().numpy(), tw.cpu().numpy()
    for l, (s, spec) in enumerate(zip(shapes, specs)):
        ok = np.ones(T, bool)
        if s.n_experts:
            lg, oidx, ow = oracle_routes(orc, spec, xt[:, l])
            ok = check_routing(gi[:, l, :s.top_k], gw[:, l, :s.top_k], lg, oidx, ow, s.top_k)
            Lo = oracle_layer(orc, spec, experts=np.unique(oidx), gen_device=DEV)
        else:
            Lo = oracle_layer(orc, spec, gen_device=DEV)
        oout, _, _ = orc.moe_forward(Lo, xt[:, l], residual=ht[:, l])
        nxt = ht[:, l + 1] if l + 1 < L else g_out
        assert_close((nxt - ht[:, l])[ok], (oout - ht[:, l])[ok], "layer %d (%s) delta" % (
            l, "dense" if not s.n_experts else "MoE"))


def test_decode_flint_dense_layers_around_moe(orc):
    # dense (6144) -> MoE -> dense, as the model's dense layers sit among its MoE layers
    _chain(orc, [synth.FLINT_DENSE, synth.FLINT, synth.FLINT_DENSE], T=3, seed=61)


def test_decode_small_dense_chain(orc):
    # a width that is not a power of two (384 = 3 parts of 128) and a dense-only chain
    _chain(orc, [SMALL_DENSE, SMALL_DENSE], T=4, seed=62)
    _chain(orc, [SMALL_DENSE, synth.TINY, SMALL_DENSE], T=4, seed=63)
