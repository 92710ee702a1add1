"""The benchmarked configurations against the oracle.

* The decode weight stream the bench times: one flint_decode_tokens launch over 47
  chained Flint layers (hidden 2048, 256 experts top-6 with a Zipf(1.1) router bias,
  width 512, shared 1024, RMSNorm eps 1e-6) and the 150,144-row NVFP4 head, on the
  bench's own seeded weights and its first four tokens.  Every layer is checked
  teacher-forced (the oracle layer fed the kernel's own per-layer input x_l and
  residual h_l, read back through flint_decode_tokens_trace); the head logits and argmax
  against the oracle head on the kernel's final x; and a free-running oracle chain from
  the token inputs alone.  The two chains' residuals differ by fp32-level rounding
  (about 1e-7 per layer); x is rounded to bf16 between layers, so once such a
  difference moves one element of x across a bf16 rounding boundary (each such step
  moves the next residual by about 1e-5) the chains part and the differences compound
  from layer to layer.  The free-running comparison therefore follows a token while the
  kernel's x_l is bit-identical to the oracle's: there its residual must agree at the
  stated tolerance and its expert set exactly (outside near-ties), and a token followed
  through all 47 layers is compared on its final residual, logits and argmax.
* One Flint layer over 1,000 seeded tokens (batch 1, one token after another): routing
  and outputs of every token.
"""
import numpy as np
import pytest
import torch

from helpers import (TIE_GAP, assert_close, bits16, check_routing, float_errors, oracle_layer,
                     oracle_routes, routing_exempt)
from sparse_moe_decode_02_b300 import flint, synth, workload

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flint.lib()


def _bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _assert_rmsnorm_inputs(orc, h: np.ndarray, x_bits: np.ndarray, what: str):
    """x = bf16(RMSNorm(h)) within one bf16 step (the reduction order may move a value
    across a rounding boundary)."""
    for t in range(h.shape[0]):
        ref = _bf16_values(orc.rmsnorm_bf16(h[t], EPS))
        got = _bf16_values(x_bits[t])
        step = np.maximum(np.abs(ref), 1e-30) * 2.0 ** -7
        assert np.all(np.abs(got - ref) <= step * 1.0001), "%s token %d" % (what, t)


def test_decode_bench_config_47_layers_and_head(orc):
    shape = synth.FLINT
    H, k, V, L, T, seed = shape.hidden, shape.top_k, shape.vocab, 47, 4, 0
    specs = [synth.LayerSpec(shape, seed=seed, layer=l, zipf=1.1) for l in range(L)]
    layers = [workload.build_layer(s, DEV) for s in specs]
    head = workload.build_head(seed, V, H, DEV)
    x = synth.tokens_bf16(seed, H, T, stream=1)               # the bench's first tokens
    f32 = dict(dtype=torch.float32, device=DEV)
    out = torch.empty(T, H, **f32)
    x_out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    logits = torch.empty(T, V, **f32)
    am = torch.empty(T, dtype=torch.int32, device=DEV)
    tidx = torch.empty(T, L, k, dtype=torch.int32, device=DEV)
    tw = torch.empty(T, L, k, **f32)
    xt = torch.empty(T, L, H, dtype=torch.bfloat16, device=DEV)
    ht = torch.empty(T, L, H, **f32)
    flint.decode_tokens(layers, x.to(DEV), head=head, rms_eps=EPS, out=out, x_out=x_out,
                        logits=logits, argmax=am, topk_idx=tidx, topk_w=tw, x_trace=xt,
                        h_trace=ht)
    torch.cuda.synchronize()
    assert flint.last_device_status() == 0
    del layers
    xt, ht = bits16(xt), ht.cpu().numpy().astype(np.float64)
    gi, gw = tidx.cpu().numpy(), tw.cpu().numpy()
    g_out = out.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(xt[:, 0], bits16(x))
    np.testing.assert_array_equal(ht[:, 0], _bf16_values(bits16(x)))

    # free-running oracle chain, followed while it sees the kernel's x bit for bit
    fx, fh = bits16(x), _bf16_values(bits16(x))
    followed = np.ones(T, bool)
    parted = {}
    for l in range(L):
        # teacher forcing: the oracle layer on the kernel's own input of layer l
        lg, oidx, ow = oracle_routes(orc, specs[l], xt[:, l])
        ok = check_routing(gi[:, l], gw[:, l], lg, oidx, ow, k)
        flg, fidx, _ = oracle_routes(orc, specs[l], fx)
        experts = np.unique(np.concatenate([oidx.ravel(), fidx.ravel()]))
        Lo = oracle_layer(orc, specs[l], experts=experts, gen_device=DEV)
        oout, _, _ = orc.moe_forward(Lo, xt[:, l], residual=ht[:, l])
        nxt = ht[:, l + 1] if l + 1 < L else g_out
        assert_close((nxt - ht[:, l])[ok], (oout - ht[:, l])[ok], "layer %d MoE delta" % l)
        if l + 1 < L:
            _assert_rmsnorm_inputs(orc, ht[:, l + 1], xt[:, l + 1], "x of layer %d" % (l + 1))
        for t in np.nonzero(followed)[0]:
            if not np.array_equal(fx[t], xt[t, l]):
                followed[t] = False
                parted[int(t)] = (l, int((fx[t] != xt[t, l]).sum()),
                                  float(float_errors(ht[t, l], fh[t])[0]))
                continue
            assert_close(ht[t, l], fh[t], "residual into layer %d, token %d (free-running)" % (l, t))
            if not routing_exempt(flg[t], k)[0]:
                np.testing.assert_array_equal(np.sort(gi[t, l]), np.sort(fidx[t]))
        fh, _, _ = orc.moe_forward(Lo, fx, residual=fh)
        fx = np.stack([orc.rmsnorm_bf16(fh[t], EPS) for t in range(T)])
    print("free-running chains parted (token: layer, x elements differing, residual rel L2):",
          parted)
    # head on the kernel's final x
    _assert_rmsnorm_inputs(orc, g_out, bits16(x_out), "head input")
    oq, st = orc.quantize_nvfp4(synth.head_bf16(seed, V, H, device=DEV).cpu())
    assert st == 0
    ol, oam = orc.lm_head(oq, bits16(x_out))
    g_lg, g_am = logits.cpu().numpy(), am.cpu().numpy()
    for t in range(T):
        assert_close(g_lg[t], ol[t], "head logits token %d" % t)
        srt = np.sort(ol[t])[::-1]
        if srt[0] - srt[1] >= TIE_GAP:
            assert int(g_am[t]) == int(oam[t])
    # end to end against the free-running oracle, for the tokens followed to the end
    fl, fam = orc.lm_head(oq, fx)
    for t in np.nonzero(followed)[0]:
        assert_close(g_out[t], fh[t], "final residual token %d (free-running oracle)" % t)
        assert_close(g_lg[t], fl[t], "logits token %d (free-running oracle)" % t)
        srt = np.sort(fl[t])[::-1]
        if srt[0] - srt[1] >= TIE_GAP:
            assert int(g_am[t]) == int(fam[t])


def test_decode_flint_layer_1000_tokens(orc):
    shape = synth.FLINT
    H, k, T = shape.hidden, shape.top_k, 1000
    spec = synth.LayerSpec(shape, seed=0, layer=0)
    layer = workload.build_layer(spec, DEV)
    x = synth.tokens_bf16(0, H, T, stream=2)
    out = torch.empty(T, H, dtype=torch.float32, device=DEV)
    tidx = torch.empty(T, 1, k, dtype=torch.int32, device=DEV)
    tw = torch.empty(T, 1, k, dtype=torch.float32, device=DEV)
    flint.decode_tokens([layer], x.to(DEV), out=out, topk_idx=tidx, topk_w=tw)
    torch.cuda.synchronize()
    assert flint.last_device_status() == 0
    xb = bits16(x)
    lg, oidx, ow = oracle_routes(orc, spec, xb)
    ok = check_routing(tidx[:, 0].cpu().numpy(), tw[:, 0].cpu().numpy(), lg, oidx, ow, k)
    assert ok.sum() >= T - 10
    Lo = oracle_layer(orc, spec, experts=np.unique(oidx), gen_device=DEV)
    oout, _, _ = orc.moe_forward(Lo, xb)
    xd = _bf16_values(xb)
    g = out.cpu().numpy().astype(np.float64)
    for t in np.nonzero(ok)[0]:
        assert_close(g[t] - xd[t], oout[t] - xd[t], "token %d MoE delta" % t)
