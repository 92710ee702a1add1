"""Pins for the oracle's NVFP4 quantiser: exact round trip of on-grid weights, the
per-element error bound that follows from the format, the special cases, and an
independent numpy restatement of the recipe.  CPU only."""
import numpy as np
import pytest
import torch

import indep

E2M1_MAGS = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_on_grid_round_trip_exact(orc):
    """Weights built as e2m1 * s * tsc with amax_b = 6 s tsc quantise back to the same
    codes and scales, and dequantise to themselves bit for bit."""
    rng = np.random.default_rng(3)
    rows, cols = 24, 64
    tsc = 2.0 ** -10
    # block scales: e4m3 values, block amax element set to 6
    sc_codes = rng.integers(0x20, 0x7E, size=(rows, cols // 16)).astype(np.uint8)
    sc_codes[0, 0] = 0x7E                                  # one block at 448 -> amax = 2688 tsc
    sc_vals = indep.e4m3_torch(sc_codes.reshape(-1)).reshape(rows, cols // 16)
    codes = rng.integers(0, 16, size=(rows, cols)).astype(np.uint8)
    codes[:, ::16] = 7                                     # each block holds a +6
    vals = np.array([indep.e2m1_closed_form(c) for c in codes.reshape(-1)]).reshape(rows, cols)
    w = vals * np.repeat(sc_vals, 16, axis=1) * tsc
    wt = torch.from_numpy(w).to(torch.bfloat16)
    assert np.array_equal(wt.double().numpy(), w), "construction must be bf16-exact"
    q, st = orc.quantize_nvfp4(wt[None])
    assert st == 0
    assert q.tsc[0] == np.float32(tsc)
    np.testing.assert_array_equal(q.scales[0], sc_codes)
    # -0 codes (8) and 0 are both exact zeros; compare values, then nibbles where non-zero
    want_packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    got = q.codes[0]
    nz = vals != 0
    got_n = np.stack([got & 15, got >> 4], -1).reshape(rows, cols)
    want_n = np.stack([want_packed & 15, want_packed >> 4], -1).reshape(rows, cols)
    np.testing.assert_array_equal(got_n[nz], want_n[nz])
    np.testing.assert_array_equal(q.dequantize()[0].astype(np.float64), w)


def _gap_bound(v):
    """Largest rounding error of E2M1 RNE+satfinite at |v| (units of the block scale)."""
    a = np.abs(v)
    half_gap = np.where(a <= 2.0, 0.25, np.where(a <= 4.0, 0.5, 1.0))
    return np.where(a > 6.0, a - 6.0, half_gap)


def test_error_bound_random(orc):
    """|w - deq(w)| <= half the E2M1 gap at |w|/eff (or the saturation excess), in units
    of eff = e4m3(amax_b/6/tsc) * tsc; and eff lies within one e4m3 rounding of
    amax_b / 6."""
    g = torch.Generator().manual_seed(4)
    w = (torch.randn(3, 40, 256, generator=g) * 0.02).to(torch.bfloat16)
    w[1] *= 1000
    w[2, :, :16] = 0          # an all-zero block
    q, st = orc.quantize_nvfp4(w)
    assert st == 0
    deq = q.dequantize().astype(np.float64)
    wd = w.double().numpy()
    n, r, c = wd.shape
    sc = indep.e4m3_torch(q.scales.reshape(-1)).reshape(n, r, c // 16)
    eff = np.repeat(sc, 16, axis=-1) * q.tsc[:, None, None].astype(np.float64)
    err = np.abs(wd - deq)
    v = np.divide(wd, eff, out=np.zeros_like(wd), where=eff > 0)
    bound = _gap_bound(v) * eff * (1 + 2.0 ** -20) + 1e-30
    assert np.all(err <= bound + np.abs(deq) * 2.0 ** -23)
    amax_b = np.abs(wd).reshape(n, r, c // 16, 16).max(-1)
    eff_b = sc * q.tsc[:, None, None]
    ok = amax_b > 0
    rel = np.abs(eff_b[ok] - amax_b[ok] / 6) / (amax_b[ok] / 6)
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)
    # the zero block
    assert np.all(q.scales[2, :, 0] == 0) and np.all(deq[2, :, :16] == 0)
    # tensor scale = amax / 2688 in fp32
    for m in range(n):
        assert q.tsc[m] == np.float32(np.float32(np.abs(wd[m]).max()) / np.float32(2688.0))


def test_independent_restatement_bit_exact(orc):
    """The recipe restated with numpy fp32 steps, torch's e4m3 cast and rint rounding."""
    g = torch.Generator().manual_seed(5)
    w = (torch.randn(2, 17, 128, generator=g) * 0.02).to(torch.bfloat16)
    q, st = orc.quantize_nvfp4(w)
    wf = w.float().numpy()
    n, r, c = wf.shape
    for m in range(n):
        amax = np.float32(np.abs(wf[m]).max())
        tsc = np.float32(amax / np.float32(2688.0))
        assert q.tsc[m] == tsc
        blocks = wf[m].reshape(r, c // 16, 16)
        amax_b = np.abs(blocks).max(-1).astype(np.float32)
        t = (amax_b / np.float32(6.0)).astype(np.float32)
        t = (t / tsc).astype(np.float32)
        s = torch.from_numpy(np.minimum(t, 448.0)).to(torch.float8_e4m3fn)
        np.testing.assert_array_equal(q.scales[m], s.view(torch.uint8).numpy())
        eff = (s.float().numpy() * tsc).astype(np.float32)
        vq = (blocks / eff[..., None]).astype(np.float32)
        code_vals = indep.e2m1_round(vq.astype(np.float64))          # E2M1 values
        # dequantised value: fp32(fp32(e2m1 * e4m3) * tsc)
        prod = (code_vals * s.double().numpy()[..., None]).astype(np.float32)
        want = (prod * tsc).astype(np.float32).reshape(r, c)
        np.testing.assert_array_equal(q.dequantize()[m], want)


def test_zero_matrix_and_nonfinite(orc):
    z = torch.zeros(1, 8, 32, dtype=torch.bfloat16)
    q, st = orc.quantize_nvfp4(z)
    assert st == 0 and q.tsc[0] == 1.0
    assert not q.codes.any() and not q.scales.any()
    bad = torch.zeros(2, 8, 32, dtype=torch.bfloat16)
    bad[1, 3, 5] = float("nan")
    _, st = orc.quantize_nvfp4(bad)
    assert st == 5
    bad[1, 3, 5] = float("inf")
    _, st = orc.quantize_nvfp4(bad)
    assert st == 5


def test_nibble_order_and_density(orc):
    """Element 2j in the low nibble of byte j; 2,048 values take 1,024 code bytes
    (the 4-bit head row size printed on the pages) plus 128 scale bytes."""
    w = torch.zeros(1, 1, 2048, dtype=torch.bfloat16)
    w[0, 0, 0] = 6.0 * 0.01   # code 7 in the low nibble of byte 0
    w[0, 0, 3] = -3.0 * 0.01  # element 3: high nibble of byte 1
    q, _ = orc.quantize_nvfp4(w)
    assert q.codes.shape == (1, 1, 1024) and q.scales.shape == (1, 1, 128)
    assert q.codes[0, 0, 0] & 15 == 7 and q.codes[0, 0, 0] >> 4 == 0
    assert q.codes[0, 0, 1] >> 4 == 13   # -3 = sign | code 5


def test_unit_scale_rows(orc):
    """Activation quantisation (tensor scale fixed at 1) equals the recipe with tsc=1."""
    rng = np.random.default_rng(6)
    v = rng.standard_normal((5, 64)).astype(np.float32)
    codes, scales = orc.quantize_rows_unit(v)
    amax_b = np.abs(v.reshape(5, 4, 16)).max(-1).astype(np.float32)
    s = torch.from_numpy((amax_b / np.float32(6.0)).astype(np.float32)).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(scales, s.view(torch.uint8).numpy())
    deq = indep.dequantize_np(codes[None], scales[None], np.ones(1, np.float32))[0]
    eff = np.repeat(s.float().numpy(), 16, axis=-1).reshape(5, 64)
    want = indep.e2m1_round((v / eff).astype(np.float32).astype(np.float64)) * eff
    np.testing.assert_array_equal(deq.astype(np.float64), want)
