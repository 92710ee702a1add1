"""Pins for the oracle's router, MoE layer, RMSNorm, output head and expert order:
brute force on tiny sizes, closed forms, invariants, and an independent numpy
restatement (library matmul over independently decoded weights).  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit, softmax

import indep
from sparse_moe_decode_02_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "flint_page_figures.json")


def _tiny_layer(orc, seed=0, E=8, k=2, H=64, F=32, Fs=48, bias=False, scale=0.02):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: (torch.randn(*s, generator=g) * scale).to(torch.bfloat16)
    rw = mk(E, H)
    gate, _ = orc.quantize_nvfp4(mk(E, F, H))
    up, _ = orc.quantize_nvfp4(mk(E, F, H))
    down, _ = orc.quantize_nvfp4(mk(E, H, F))
    sg, _ = orc.quantize_nvfp4(mk(1, Fs, H))
    su, _ = orc.quantize_nvfp4(mk(1, Fs, H))
    sd, _ = orc.quantize_nvfp4(mk(1, H, Fs))
    b = (torch.randn(E, generator=g).numpy().astype(np.float32) if bias else None)
    return orc.Layer(rw, b, gate, up, down, sg, su, sd, k)


def _x(n, H, seed=1):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(n, H, generator=g).to(torch.bfloat16)


def _numpy_forward(L, x_bits, quantize_acts=False, orc=None, sigmoid=False):
    """Independent restatement: numpy matmul over weights decoded by indep."""
    deq = lambda m: indep.dequantize_np(m.codes, m.scales, m.tsc).astype(np.float64)
    Wg, Wu, Wd = deq(L.gate), deq(L.up), deq(L.down)
    Sg, Su, Sd = deq(L.sh_gate)[0], deq(L.sh_up)[0], deq(L.sh_down)[0]
    Wr = indep.bf16_to_f64(L.router_w)
    xs = indep.bf16_to_f64(x_bits)
    outs, idxs, ws = [], [], []
    for x in xs:
        logits = Wr @ x + (0 if L.router_bias is None else L.router_bias.astype(np.float64))
        order = np.argsort(-logits, kind="stable")[:L.top_k]
        w = (expit(logits[order]) / expit(logits[order]).sum() if sigmoid
             else softmax(logits[order]))
        xin = x
        if quantize_acts:
            xin = _requant(orc, x)
        out = x.copy()
        for e, we in zip(order, w):
            h = (Wg[e] @ xin) * expit(Wg[e] @ xin) * (Wu[e] @ xin)
            if quantize_acts:
                h = _requant(orc, h)
            out += we * (Wd[e] @ h)
        hs = (Sg @ xin) * expit(Sg @ xin) * (Su @ xin)
        if quantize_acts:
            hs = _requant(orc, hs)
        out += Sd @ hs
        outs.append(out); idxs.append(order); ws.append(w)
    return np.array(outs), np.array(idxs), np.array(ws)


def _requant(orc, v):
    codes, scales = orc.quantize_rows_unit(v.astype(np.float32)[None])
    return indep.dequantize_np(codes[None], scales[None], np.ones(1, np.float32))[0, 0].astype(
        np.float64)


def test_router_topk_bruteforce_and_weights(orc):
    """For E <= 8, the selected set is the size-k subset with the largest logit sum
    (logits distinct), ordered by logit; weights are the softmax over the selected
    logits alone and sum to 1."""
    for seed in range(6):
        for E, k in [(4, 1), (5, 2), (8, 3), (8, 8), (6, 6)]:
            L = _tiny_layer(orc, seed=seed, E=E, k=k, H=32, F=16, Fs=16, bias=seed % 2 == 1)
            x = _x(1, 32, seed=10 + seed)
            logits, idx, w = orc.router(L, x)
            best = max(itertools.combinations(range(E), k), key=lambda s: sum(logits[i] for i in s))
            assert sorted(idx.tolist()) == sorted(best)
            assert all(logits[idx[i]] >= logits[idx[i + 1]] for i in range(k - 1))
            np.testing.assert_allclose(w, softmax(logits[idx]), rtol=1e-13)
            assert abs(w.sum() - 1.0) < 1e-12
            # logits are the bf16 matvec (+ bias)
            want = indep.bf16_to_f64(L.router_w) @ indep.bf16_to_f64(x.view(torch.int16).numpy().view(np.uint16)[0])
            if L.router_bias is not None:
                want = want + L.router_bias
            np.testing.assert_allclose(logits, want, rtol=1e-12, atol=1e-15)


def _with_score(orc, L, score, router_w=None, bias=None):
    return orc.Layer(L.router_w if router_w is None else router_w,
                     L.router_bias if bias is None else bias, L.gate, L.up, L.down, L.sh_gate,
                     L.sh_up, L.sh_down, L.top_k, router_score=score)


def test_router_sigmoid_bruteforce_and_weights(orc):
    """Sigmoid scoring: the selected set is the size-k subset with the largest sum of
    sigmoid scores, ordered by score; weights are the selected scores over their sum;
    the set is the one softmax scoring selects (sigmoid is increasing)."""
    for seed in range(6):
        for E, k in [(4, 1), (5, 2), (8, 3), (8, 8), (6, 6)]:
            L = _tiny_layer(orc, seed=seed, E=E, k=k, H=32, F=16, Fs=16, bias=seed % 2 == 1)
            Ls = _with_score(orc, L, orc.ROUTER_SIGMOID)
            x = _x(1, 32, seed=10 + seed)
            logits, idx, w = orc.router(Ls, x)
            sc = expit(logits)
            best = max(itertools.combinations(range(E), k), key=lambda st: sum(sc[i] for i in st))
            assert sorted(idx.tolist()) == sorted(best)
            assert all(sc[idx[i]] >= sc[idx[i + 1]] for i in range(k - 1))
            np.testing.assert_allclose(w, sc[idx] / sc[idx].sum(), rtol=1e-13)
            assert abs(w.sum() - 1.0) < 1e-12
            _, idx_soft, _ = orc.router(L, x)
            np.testing.assert_array_equal(idx, idx_soft)


def test_router_sigmoid_closed_form(orc):
    """Zero router weights make the logits equal the bias.  Logits 0, ln 3, -ln 3 score
    1/2, 3/4, 1/4, so top-2 picks experts 1 then 0 with weights 3/5 and 2/5; with all
    logits equal every selected expert gets 1/k."""
    L = _tiny_layer(orc, E=4, k=2, H=32, F=16, Fs=16)
    zero = np.zeros_like(L.router_w)
    ln3 = math.log(3.0)
    Ls = _with_score(orc, L, orc.ROUTER_SIGMOID, router_w=zero,
                     bias=np.array([0.0, ln3, -ln3, -2 * ln3], np.float32))
    logits, idx, w = orc.router(Ls, _x(1, 32))
    np.testing.assert_array_equal(idx, [1, 0])
    np.testing.assert_allclose(w, [0.6, 0.4], rtol=1e-7)
    Le = _with_score(orc, L, orc.ROUTER_SIGMOID, router_w=zero,
                     bias=np.full(4, 0.7, np.float32))
    _, idx, w = orc.router(Le, _x(1, 32))
    np.testing.assert_array_equal(idx, [0, 1])          # ties to the lower index
    np.testing.assert_allclose(w, [0.5, 0.5], rtol=1e-15)


def test_layer_sigmoid_matches_numpy_restatement(orc):
    L = _with_score(orc, _tiny_layer(orc, seed=4, E=8, k=3, H=64, F=32, Fs=48, bias=True),
                    orc.ROUTER_SIGMOID)
    x = _x(5, 64, seed=6)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    out, idx, w = orc.moe_forward(L, x)
    ref, ridx, rw = _numpy_forward(L, xb, sigmoid=True)
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=1e-12)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)


def test_router_ties_go_to_lower_index(orc):
    E, H = 8, 16
    L = _tiny_layer(orc, E=E, k=3, H=H, F=16, Fs=16)
    # identical router rows 1, 4, 6: equal logits
    rw = L.router_w.copy()
    rw[1] = rw[1] & 0x7FFF          # |row 1| (clear the bf16 sign bits): the largest logit
    rw[4] = rw[1]; rw[6] = rw[1]
    L2 = orc.Layer(rw, None, L.gate, L.up, L.down, L.sh_gate, L.sh_up, L.sh_down, 3)
    x = torch.ones(1, H, dtype=torch.bfloat16)
    logits, idx, w = orc.router(L2, x)
    assert logits[1] == logits[4] == logits[6]
    stable = np.argsort(-logits, kind="stable")[:3]
    np.testing.assert_array_equal(idx, stable)


def test_layer_matches_numpy_restatement(orc):
    for bias in (False, True):
        L = _tiny_layer(orc, seed=2, E=8, k=3, H=64, F=32, Fs=48, bias=bias)
        x = _x(5, 64, seed=3)
        xb = x.view(torch.int16).numpy().view(np.uint16)
        out, idx, w = orc.moe_forward(L, x)
        ref, ridx, rw = _numpy_forward(L, xb)
        np.testing.assert_array_equal(idx, ridx)
        np.testing.assert_allclose(w, rw, rtol=1e-12)
        np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)


def test_prefill_mode_matches_numpy_restatement(orc):
    L = _tiny_layer(orc, seed=4, E=8, k=2, H=64, F=32, Fs=32)
    x = _x(4, 64, seed=5)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    out, idx, _ = orc.moe_forward(L, x, quantize_acts=True)
    ref, ridx, _ = _numpy_forward(L, xb, quantize_acts=True, orc=orc)
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12)
    # and it stays close to the unquantised layer (activation quantisation error only)
    plain, _, _ = orc.moe_forward(L, x)
    xd = indep.bf16_to_f64(xb)
    rel = np.linalg.norm((out - xd) - (plain - xd)) / np.linalg.norm(plain - xd)
    assert rel < 0.2


def test_shared_expert_always_contributes(orc):
    """Zero routed down weights -> out = x + shared(x); zero shared down -> out - x is the
    routed part only."""
    L = _tiny_layer(orc, seed=6)
    x = _x(3, 64, seed=7)
    zero_down = orc.NVFP4(np.zeros_like(L.down.codes), np.zeros_like(L.down.scales), L.down.tsc)
    Lr0 = orc.Layer(L.router_w, None, L.gate, L.up, zero_down, L.sh_gate, L.sh_up, L.sh_down, 2)
    out_r0, _, _ = orc.moe_forward(Lr0, x)
    zero_sd = orc.NVFP4(np.zeros_like(L.sh_down.codes), np.zeros_like(L.sh_down.scales),
                        L.sh_down.tsc)
    Ls0 = orc.Layer(L.router_w, None, L.gate, L.up, L.down, L.sh_gate, L.sh_up, zero_sd, 2)
    out_s0, _, _ = orc.moe_forward(Ls0, x)
    full, _, _ = orc.moe_forward(L, x)
    xd = indep.bf16_to_f64(x.view(torch.int16).numpy().view(np.uint16))
    assert np.abs(out_r0 - xd).max() > 0            # the shared expert always adds something
    np.testing.assert_allclose((out_r0 - xd) + (out_s0 - xd), full - xd, rtol=1e-12, atol=1e-15)


def test_k_equals_e_is_dense_softmax_mixture(orc):
    E = 6
    L = _tiny_layer(orc, seed=8, E=E, k=E, H=32, F=16, Fs=16)
    x = _x(2, 32, seed=9)
    out, idx, w = orc.moe_forward(L, x)
    logits = [orc.router(L, x[i:i + 1])[0] for i in range(2)]
    xd = indep.bf16_to_f64(x.view(torch.int16).numpy().view(np.uint16))
    for t in range(2):
        p = softmax(logits[t])
        np.testing.assert_allclose(np.sort(w[t]), np.sort(p), rtol=1e-12)
        # sum_e p_e * expert_e(x): build it with single-expert layers (k = 1, forced
        # selection through a large bias on expert e)
        mix = np.zeros(32)
        for e in range(E):
            bias = np.full(E, -1e4, np.float32); bias[e] = 0
            Le = orc.Layer(L.router_w, bias, L.gate, L.up, L.down, L.sh_gate, L.sh_up, L.sh_down, 1)
            oe, ie, _ = orc.moe_forward(Le, x[t:t + 1])
            assert ie[0, 0] == e
            mix += p[e] * oe[0]
        # each single-expert output carries x + shared once; the p_e sum to 1
        np.testing.assert_allclose(out[t], mix, rtol=1e-10, atol=1e-13)


def test_rmsnorm_closed_forms(orc):
    c = np.full(64, 3.0)
    y = indep.bf16_to_f64(orc.rmsnorm_bf16(c, 0.0))
    np.testing.assert_array_equal(y, np.ones(64))
    h = np.array([3.0, -4.0] * 8)
    y = indep.bf16_to_f64(orc.rmsnorm_bf16(h, 1e-6))
    r = 1 / math.sqrt(12.5 + 1e-6)
    want = torch.tensor(h * r, dtype=torch.float64).to(torch.float32).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(y, want)


def test_lm_head_matches_numpy_and_argmax_ties(orc):
    g = torch.Generator().manual_seed(11)
    W, _ = orc.quantize_nvfp4((torch.randn(1, 300, 64, generator=g) * 0.02).to(torch.bfloat16))
    x = _x(3, 64, seed=12)
    logits, am = orc.lm_head(W, x)
    Wd = indep.dequantize_np(W.codes, W.scales, W.tsc)[0].astype(np.float64)
    xd = indep.bf16_to_f64(x.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_allclose(logits, xd @ Wd.T, rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(am, np.argmax(xd @ Wd.T, axis=1))
    # duplicate the winning row further down: the lower index must win
    codes = W.codes.copy(); scales = W.scales.copy()
    win = int(am[0])
    codes[0, 299] = codes[0, win]; scales[0, 299] = scales[0, win]
    codes[0, :win] = 0
    W2 = orc.NVFP4(codes, scales, W.tsc)
    l2, am2 = orc.lm_head(W2, x[:1])
    assert l2[0, 299] == l2[0, win] and am2[0] == win


def test_expert_order_is_stable_counting_sort(orc):
    rng = np.random.default_rng(13)
    idx = np.stack([rng.choice(16, 3, replace=False) for _ in range(50)]).astype(np.int32)
    counts, offsets, perm = orc.expert_order(idx, 16)
    np.testing.assert_array_equal(counts, np.bincount(idx.reshape(-1), minlength=16))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)[:-1]]))
    np.testing.assert_array_equal(perm, np.argsort(idx.reshape(-1), kind="stable"))


def test_page_byte_accounting():
    """The shapes reproduce the parameter and byte counts printed on the pages."""
    g = {k: v for k, v in json.load(open(GOLDEN)).items() if not k.startswith("_")}
    s = synth.FLINT
    assert (s.hidden, s.n_experts, s.expert_width, s.top_k, s.shared_width, s.vocab) == (
        g["hidden"]["value"], g["routed_experts"]["value"], g["expert_width"]["value"],
        g["top_k"]["value"], g["shared_width"]["value"], g["vocab"]["value"])
    layers = g["moe_layers"]["value"]
    per_expert = 3 * s.hidden * s.expert_width
    total = layers * s.n_experts * per_expert
    per_tok = layers * s.top_k * per_expert
    head = s.vocab * s.hidden
    rel = lambda a, b, t: abs(a - b) / b <= t
    assert rel(total, g["routed_params_total"]["value"], g["routed_params_total"]["rel_tol"])
    assert rel(per_tok, g["routed_params_per_token"]["value"], g["routed_params_per_token"]["rel_tol"])
    assert rel(head, g["head_params"]["value"], g["head_params"]["rel_tol"])
    bpw = (4 + 8 / g["block"]["value"]) / 8          # 4-bit value + 8-bit scale per 16
    assert bpw * 8 == g["bits_per_weight"]["value"]
    assert abs(per_tok * bpw / 1e6 - g["routed_mb_per_token_4p5bpw"]["value"]) <= 0.5
    assert abs(head * bpw / 1e6 - g["head_mb_per_token_4p5bpw"]["value"]) <= 0.5
    assert s.hidden * 4 // 8 == g["head_bytes_per_row_4bit"]["value"]


def _dense_layer(orc, seed=5, H=64, Fs=384, scale=0.02):
    """A dense SwiGLU layer (no router, no routed experts; the block in sh_*)."""
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: (torch.randn(*s, generator=g) * scale).to(torch.bfloat16)
    empty = lambda r, c: orc.NVFP4(np.zeros((0, r, c // 2), np.uint8), np.zeros((0, r, c // 16), np.uint8),
                                   np.zeros(0, np.float32))
    sg, _ = orc.quantize_nvfp4(mk(1, Fs, H))
    su, _ = orc.quantize_nvfp4(mk(1, Fs, H))
    sd, _ = orc.quantize_nvfp4(mk(1, H, Fs))
    return orc.Layer(np.zeros((0, H), np.uint16), None, empty(0, H), empty(0, H), empty(H, 0), sg, su, sd, 0)


def test_dense_layer_matches_numpy_restatement(orc):
    # out = residual + Wd (silu(Wg x) * (Wu x)): the block alone, no router (width 384 is
    # not a power of two, as the model's 6,144 is not)
    L = _dense_layer(orc)
    xb = orc._bits16(_x(5, 64, seed=9))
    res = np.random.default_rng(3).standard_normal((5, 64))
    out, idx, w = orc.moe_forward(L, xb, residual=res)
    deq = lambda m: indep.dequantize_np(m.codes, m.scales, m.tsc).astype(np.float64)[0]
    Sg, Su, Sd = deq(L.sh_gate), deq(L.sh_up), deq(L.sh_down)
    xs = indep.bf16_to_f64(xb)
    want = res + np.stack([Sd @ (indep.silu(Sg @ x) * (Su @ x)) for x in xs])
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)
    assert idx.shape == (5, 0) and w.shape == (5, 0)


def test_dense_layer_zero_down_is_identity(orc):
    L = _dense_layer(orc, seed=6)
    zero, _ = orc.quantize_nvfp4(torch.zeros(1, 64, 384, dtype=torch.bfloat16))
    L.sh_down = zero
    xb = orc._bits16(_x(3, 64, seed=10))
    out, _, _ = orc.moe_forward(L, xb)
    np.testing.assert_array_equal(out, indep.bf16_to_f64(xb))
