"""Independent routes to the quantities the oracle computes, used only to pin it.

Nothing here calls the oracle.  The number formats are rebuilt from their closed
forms, or from a library routine (torch's float8_e4m3fn cast), and the rounding
to a mini-float grid uses numpy's round-half-even (``np.rint``) on a rescaled
value instead of the oracle's table search.
"""
from __future__ import annotations

import numpy as np
import torch


def e2m1_closed_form(code: int) -> float:
    """(-1)^s * (e == 0 ? m/2 : 2^(e-1) * (1 + m/2)), fields s|e1 e0|m."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1.0 + m / 2.0)
    return -mag if s else mag


def e4m3_torch(byte_vals) -> np.ndarray:
    """Decode E4M3 bytes with torch's float8_e4m3fn dtype."""
    b = torch.as_tensor(np.asarray(byte_vals, dtype=np.uint8))
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def round_minifloat(v, mant_bits: int, emin: int, vmax: float) -> np.ndarray:
    """Round to a binary mini-float (mant_bits stored mantissa bits, minimum normal
    exponent emin, largest finite vmax), half to even, saturating to +-vmax."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    quantum = np.exp2(e - mant_bits)
    q = np.rint(a / quantum) * quantum      # np.rint: round half to even
    q = np.minimum(q, vmax)
    return np.copysign(q, v)


def e2m1_round(v):
    return round_minifloat(v, mant_bits=1, emin=0, vmax=6.0)


def e4m3_round(v):
    return round_minifloat(v, mant_bits=3, emin=-6, vmax=448.0)


_E2M1_VALS = np.array([e2m1_closed_form(c) for c in range(16)])


def dequantize_np(codes: np.ndarray, scales: np.ndarray, tsc: np.ndarray) -> np.ndarray:
    """codes [n, R, C/2], scales [n, R, C/16], tsc [n] -> fp32 [n, R, C]:
    fp32(fp32(e2m1 * e4m3) * tsc), decoded with the closed form and torch."""
    n, r, half = codes.shape
    lo = codes & 0xF
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(n, r, half * 2)
    val = _E2M1_VALS[nib]
    sc = e4m3_torch(scales.reshape(-1)).reshape(scales.shape)
    sc_full = np.repeat(sc, 16, axis=-1)
    prod = (val * sc_full).astype(np.float32)
    return (prod * tsc.astype(np.float32)[:, None, None]).astype(np.float32)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def silu(g):
    return g / (1.0 + np.exp(-g))
