"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on the same
seeded inputs.  Quantisation bytes and dequantised values bit-exact; routing exact
outside near-ties; floats within relative L2 2e-3 and max-abs 1e-2 x RMS."""
import numpy as np
import pytest
import torch

from helpers import (assert_close, bits16, check_routing, oracle_layer, oracle_routes,
                     TIE_GAP)
from sparse_moe_decode_02_b300 import flint, synth, workload

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flint.lib()


def _assert_quant_equal(gq, oq, what):
    np.testing.assert_array_equal(gq.tsc.cpu().numpy().view(np.uint32),
                                  oq.tsc.view(np.uint32), err_msg=what + " tensor scale")
    np.testing.assert_array_equal(gq.scales.cpu().numpy(), oq.scales, err_msg=what + " scales")
    np.testing.assert_array_equal(gq.codes.cpu().numpy(), oq.codes, err_msg=what + " codes")


# ------------------------------------------------------------------ quantiser
@pytest.mark.parametrize("shape", [(3, 40, 256), (1, 7, 2048), (2, 64, 96)])
def test_quantize_bitexact_random(orc, shape):
    key = synth.tensor_key(7, *shape)
    n = int(np.prod(shape))
    w = synth.normal_bf16(key, n, 0.02).view(*shape)
    w[0, 0, :16] = 0                                # an all-zero block
    w[-1, -1, :5] = torch.tensor([1e-30, -1e-30, -0.0, 3e-3, -2e-3])
    if shape[0] > 1:
        w[1] *= 3000                                 # a second tensor scale range
    gq = flint.quantize_nvfp4(w.to(DEV))
    oq, st = orc.quantize_nvfp4(w)
    assert st == 0
    _assert_quant_equal(gq, oq, "quantize %s" % (shape,))
    assert flint.last_device_status() == 0


def test_quantize_bitexact_ties_and_grid(orc):
    """On-grid values, exact E2M1 midpoints and saturation cases."""
    rng = np.random.default_rng(0)
    rows, cols = 32, 64
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5, 5.9])
    vals = rng.choice(mags, size=(rows, cols)) * rng.choice([-1, 1], size=(rows, cols))
    vals[:, ::16] = 6.0
    sc = 2.0 ** rng.integers(-8, 4, size=(rows, cols // 16))
    w = torch.from_numpy(vals * np.repeat(sc, 16, axis=1) * 2.0 ** -6).to(torch.bfloat16)[None]
    gq = flint.quantize_nvfp4(w.to(DEV))
    oq, _ = orc.quantize_nvfp4(w)
    _assert_quant_equal(gq, oq, "grid/ties")


def test_dequantize_bitexact(orc):
    w = synth.normal_bf16(synth.tensor_key(8), 5 * 64 * 512, 0.02).view(5, 64, 512)
    oq, _ = orc.quantize_nvfp4(w)
    gq = flint.NVFP4(torch.from_numpy(oq.codes).to(DEV), torch.from_numpy(oq.scales).to(DEV),
                     torch.from_numpy(oq.tsc).to(DEV))
    got = flint.dequantize_nvfp4(gq).cpu().numpy()
    np.testing.assert_array_equal(got.view(np.uint32), oq.dequantize().view(np.uint32))


def test_quantize_nonfinite_sets_status():
    w = torch.zeros(2, 8, 32, dtype=torch.bfloat16, device=DEV)
    w[1, 2, 3] = float("nan")
    flint.last_device_status()
    flint.quantize_nvfp4(w)
    assert flint.last_device_status() == 5
    assert flint.last_device_status() == 0          # read clears


# ------------------------------------------------------------------ decode
def _decode_case(orc, spec, x_bits_t, B, residual=None):
    """Runs the GPU layer on x (T tokens, B at a time) and the oracle on the same."""
    T = x_bits_t.shape[0]
    layer = workload.build_layer(spec, DEV)
    k = spec.shape.top_k
    x_bits = bits16(x_bits_t)
    logits, oidx, ow = oracle_routes(orc, spec, x_bits)
    L = oracle_layer(orc, spec, experts=np.unique(oidx))
    oout, oidx2, _ = orc.moe_forward(L, x_bits, residual=residual)
    np.testing.assert_array_equal(oidx2, oidx)
    xd = x_bits_t.to(DEV)
    out = torch.empty(T, spec.shape.hidden, dtype=torch.float32, device=DEV)
    gidx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    gw = torch.empty(T, k, dtype=torch.float32, device=DEV)
    res_d = None if residual is None else torch.from_numpy(residual.astype(np.float32)).to(DEV)
    for t0 in range(0, T, B):
        t1 = min(T, t0 + B)
        flint.moe_decode(layer, xd[t0:t1], residual=None if res_d is None else res_d[t0:t1],
                         out=out[t0:t1], topk_idx=gidx[t0:t1], topk_w=gw[t0:t1])
    torch.cuda.synchronize()
    assert flint.last_device_status() == 0
    ok = check_routing(gidx.cpu().numpy(), gw.cpu().numpy(), logits, oidx, ow, k)
    base = (x_bits_t.double().numpy() if residual is None else residual)
    g = out.cpu().numpy().astype(np.float64)
    assert_close(g[ok] - base[ok], oout[ok] - base[ok], "MoE delta (out - residual)")
    assert_close(g[ok], oout[ok], "out")
    return layer, g, oout


@pytest.mark.parametrize("B", [1, 3, 8])
def test_decode_tiny_all_tokens(orc, B):
    spec = synth.LayerSpec(synth.TINY, seed=0)
    x = synth.tokens_bf16(0, synth.TINY.hidden, 24)
    _decode_case(orc, spec, x, B)


def test_decode_tiny_bias_residual(orc):
    spec = synth.LayerSpec(synth.TINY, seed=3, zipf=1.1)
    x = synth.tokens_bf16(3, synth.TINY.hidden, 16)
    res = np.random.default_rng(1).standard_normal((16, synth.TINY.hidden))
    _decode_case(orc, spec, x, 2, residual=res)


def test_decode_tiny_sigmoid_router(orc):
    # FLINT_ROUTER_SIGMOID: the same selection, weights from the selected sigmoids
    spec = synth.LayerSpec(synth.TINY, seed=7, zipf=1.1, router_score=1)
    x = synth.tokens_bf16(7, synth.TINY.hidden, 12)
    _decode_case(orc, spec, x, 3)


def test_decode_flint_layer_sigmoid_sampled(orc):
    spec = synth.LayerSpec(synth.FLINT, seed=2, zipf=1.1, router_score=1)
    idx = [0, 500, 999]
    x = torch.cat([synth.tokens_bf16(2, synth.FLINT.hidden, 1, start_tok=t) for t in idx])
    _decode_case(orc, spec, x, 1)


def test_decode_flint_layer_sampled(orc):
    """Full-size Flint layer (hidden 2048, 256 experts, top-6, shared 1024), tokens of the
    seeded 1000-token stream checked one at a time, as the benchmark runs them."""
    spec = synth.LayerSpec(synth.FLINT, seed=0)
    idx = [0, 1, 2, 499, 998, 999]
    x = torch.cat([synth.tokens_bf16(0, synth.FLINT.hidden, 1, start_tok=t) for t in idx])
    _decode_case(orc, spec, x, 1)


def test_decode_x_next_rmsnorm(orc):
    spec = synth.LayerSpec(synth.TINY, seed=5)
    layer = workload.build_layer(spec, DEV)
    x = synth.tokens_bf16(5, synth.TINY.hidden, 4).to(DEV)
    xn = torch.empty_like(x)
    out = flint.moe_decode(layer, x, x_next=xn, rms_eps=1e-6)
    torch.cuda.synchronize()
    o = out.cpu().numpy().astype(np.float64)
    got = xn.cpu().float().numpy().astype(np.float64)
    for t in range(4):
        want = orc.rmsnorm_bf16(o[t], 1e-6)
        wantd = (want.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        # one bf16 rounding apart at most (fp32 on the GPU vs fp64 in the oracle)
        assert np.all(np.abs(got[t] - wantd) <= np.abs(wantd) * 2.0 ** -7 + 1e-30)


def test_decode_out_aliases_residual(orc):
    spec = synth.LayerSpec(synth.TINY, seed=6)
    layer = workload.build_layer(spec, DEV)
    x = synth.tokens_bf16(6, synth.TINY.hidden, 2).to(DEV)
    r = torch.randn(2, synth.TINY.hidden, device=DEV)
    want = flint.moe_decode(layer, x, residual=r.clone())
    flint.moe_decode(layer, x, residual=r, out=r)
    torch.cuda.synchronize()
    # every sum has a fixed order: bit for bit the same
    assert torch.equal(r, want)


# ------------------------------------------------------------------ lm_head
@pytest.fixture(scope="module")
def flint_head(orc):
    V, H = synth.FLINT.vocab, synth.FLINT.hidden
    w = synth.head_bf16(0, V, H)
    oq, st = orc.quantize_nvfp4(w)
    assert st == 0
    return oq


@pytest.mark.parametrize("B", [1, 8])
def test_lm_head_flint(orc, flint_head, B):
    V, H = synth.FLINT.vocab, synth.FLINT.hidden
    W = workload.build_head(0, V, H, DEV)
    _assert_quant_equal(W, flint_head, "head quantisation")
    x = synth.tokens_bf16(1, H, B, stream=2)
    logits, am = flint.lm_head(W, x.to(DEV))
    torch.cuda.synchronize()
    ol, oam = orc.lm_head(flint_head, bits16(x))
    g = logits.cpu().numpy()
    for b in range(B):
        assert_close(g[b], ol[b], "logits row %d" % b)
        srt = np.sort(ol[b])[::-1]
        if srt[0] - srt[1] >= TIE_GAP:
            assert int(am[b]) == int(oam[b])
        assert g[b, int(am[b])] == g[b].max()


def test_lm_head_tiny_ties(orc):
    """Duplicate rows: the argmax must take the lower index."""
    V, H = synth.TINY.vocab, synth.TINY.hidden
    w = synth.head_bf16(4, V, H)
    w[0, 3000] = w[0, 17]
    oq, _ = orc.quantize_nvfp4(w)
    W = flint.quantize_nvfp4(w.to(DEV))
    x = synth.tokens_bf16(9, H, 3)
    logits, am = flint.lm_head(W, x.to(DEV))
    ol, oam = orc.lm_head(oq, bits16(x))
    g = logits.cpu().numpy()
    for b in range(3):
        assert_close(g[b], ol[b], "tiny logits")
        assert g[b, 17] == g[b, 3000]
        assert int(am[b]) == int(oam[b]) or abs(np.sort(ol[b])[-1] - np.sort(ol[b])[-2]) < TIE_GAP
        assert int(am[b]) != 3000


def test_lm_head_argmax_only():
    V, H = synth.TINY.vocab, synth.TINY.hidden
    W = workload.build_head(2, V, H, DEV)
    x = synth.tokens_bf16(2, H, 2).to(DEV)
    lg, am = flint.lm_head(W, x)
    _, am2 = flint.lm_head(W, x, want_logits=False)
    torch.cuda.synchronize()
    assert torch.equal(am, am2)
    assert torch.equal(am.long(), lg.argmax(dim=1))


# ------------------------------------------------------------------ persistent multi-layer decode
def test_mma_scales_bitexact():
    w = synth.normal_bf16(synth.tensor_key(10), 2 * 256 * 512, 0.02).view(2, 256, 512).to(DEV)
    m = flint.quantize_nvfp4(w)
    sf = flint.nvfp4_mma_scales(m).cpu().numpy().reshape(2, 2, 8, 512)   # [m][row tile][k64][512]
    scales = m.scales.cpu().numpy().reshape(2, 2, 128, 8, 4)              # [m][rt][i][k64][j]
    i = np.arange(128)
    for j in range(4):
        got = sf[:, :, :, 16 * (i % 32) + 4 * (i // 32) + j]              # [m][rt][k64][i]
        np.testing.assert_array_equal(got, scales[:, :, :, :, j].transpose(0, 1, 3, 2))


def _chain_case(orc, shape, n_layers, T, seed, zipf, with_head):
    """GPU: one flint_decode_tokens launch over n_layers (+ head), and the same chain one
    layer at a time (flint_moe_decode).  Each layer of the one-at-a-time chain is checked
    against the oracle fed the GPU's own inputs (teacher forcing); the one-launch chain
    must agree with it."""
    H, k = shape.hidden, shape.top_k
    specs = [synth.LayerSpec(shape, seed=seed, layer=l, zipf=zipf) for l in range(n_layers)]
    layers = [workload.build_layer(s, DEV) for s in specs]
    head = workload.build_head(seed, shape.vocab, H, DEV) if with_head else None
    x = synth.tokens_bf16(seed, H, T, stream=3)
    xd = x.to(DEV)
    out = torch.empty(T, H, dtype=torch.float32, device=DEV)
    x_out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    am = torch.empty(T, dtype=torch.int32, device=DEV) if with_head else None
    lg = torch.empty(T, shape.vocab, dtype=torch.float32, device=DEV) if with_head else None
    tidx = torch.empty(T, n_layers, k, dtype=torch.int32, device=DEV)
    tw = torch.empty(T, n_layers, k, dtype=torch.float32, device=DEV)
    flint.decode_tokens(layers, xd, head=head, rms_eps=1e-6, out=out, x_out=x_out, logits=lg,
                        argmax=am, topk_idx=tidx, topk_w=tw)
    torch.cuda.synchronize()
    assert flint.last_device_status() == 0
    # the same chain one layer at a time, with oracle checks per layer
    h = None
    xl = xd
    for l in range(n_layers):
        o = torch.empty(T, H, dtype=torch.float32, device=DEV)
        xn = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
        gi = torch.empty(T, k, dtype=torch.int32, device=DEV)
        gw = torch.empty(T, k, dtype=torch.float32, device=DEV)
        for t0 in range(0, T, 8):
            t1 = min(T, t0 + 8)
            flint.moe_decode(layers[l], xl[t0:t1], residual=None if h is None else h[t0:t1],
                             out=o[t0:t1], x_next=xn[t0:t1], topk_idx=gi[t0:t1], topk_w=gw[t0:t1])
        torch.cuda.synchronize()
        xb = bits16(xl)
        res = None if h is None else h.cpu().numpy().astype(np.float64)
        logits, oidx, ow = oracle_routes(orc, specs[l], xb)
        L = oracle_layer(orc, specs[l], experts=np.unique(oidx))
        oout, _, _ = orc.moe_forward(L, xb, residual=res)
        ok = check_routing(gi.cpu().numpy(), gw.cpu().numpy(), logits, oidx, ow, k)
        base = xb.astype(np.uint32) << 16
        base = base.view(np.float32).astype(np.float64) if res is None else res
        g = o.cpu().numpy().astype(np.float64)
        assert_close(g[ok] - base[ok], oout[ok] - base[ok], "layer %d MoE delta" % l)
        # the one-launch chain selected the same experts at this layer
        np.testing.assert_array_equal(np.sort(tidx[:, l].cpu().numpy(), 1),
                                      np.sort(gi.cpu().numpy(), 1))
        h, xl = o, xn
    assert_close(out.cpu().numpy(), h.cpu().numpy(), "one-launch vs layer-by-layer out")
    d = (x_out.float() - xl.float()).abs().max().item()
    assert d <= 2.0 ** -6 * xl.float().abs().max().item()
    if with_head:
        oq, _ = orc.quantize_nvfp4(synth.head_bf16(seed, shape.vocab, H))
        ol, oam = orc.lm_head(oq, bits16(x_out))
        g = lg.cpu().numpy()
        for t in range(T):
            assert_close(g[t], ol[t], "head logits token %d" % t)
            srt = np.sort(ol[t])[::-1]
            if srt[0] - srt[1] >= TIE_GAP:
                assert int(am[t]) == int(oam[t])


def test_decode_tokens_tiny_chain_with_head(orc):
    _chain_case(orc, synth.TINY, n_layers=4, T=6, seed=11, zipf=1.1, with_head=True)


def test_decode_tokens_flint_chain(orc):
    _chain_case(orc, synth.FLINT, n_layers=3, T=2, seed=12, zipf=1.1, with_head=False)


def test_decode_tokens_flint_head_argmax_only():
    shape = synth.FLINT
    layers = [workload.build_layer(synth.LayerSpec(shape, seed=13, layer=0, zipf=1.1), DEV)]
    head = workload.build_head(13, shape.vocab, shape.hidden, DEV)
    x = synth.tokens_bf16(13, shape.hidden, 3, stream=4).to(DEV)
    am = torch.empty(3, dtype=torch.int32, device=DEV)
    lg = torch.empty(3, shape.vocab, dtype=torch.float32, device=DEV)
    xo = torch.empty(3, shape.hidden, dtype=torch.bfloat16, device=DEV)
    flint.decode_tokens(layers, x, head=head, x_out=xo, argmax=am, logits=lg)
    _, am2 = flint.lm_head(head, xo)
    torch.cuda.synchronize()
    assert torch.equal(am, am2)
    assert torch.equal(am.long(), lg.argmax(dim=1))
