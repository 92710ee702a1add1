"""Shared test helpers: oracle-side layers from the seeded generator, and the comparison
rules (bit-exact bytes; routing exact outside near-ties; floats by relative L2 and
max-abs against the output RMS)."""
from __future__ import annotations

import numpy as np
import torch

from oracle import seeded
from sparse_moe_decode_02_b300 import synth

REL_L2 = 2e-3          # relative L2 bound on floating outputs
MAX_ABS_FRAC = 1e-2    # max |err| <= MAX_ABS_FRAC * RMS(reference)
TIE_GAP = 1e-4         # routing / argmax decisions closer than this are exempt


def bits16(t: torch.Tensor) -> np.ndarray:
    return seeded.bits16(t)


def oracle_stack(orc, spec: synth.LayerSpec, kind: int, experts, gen_device="cpu"):
    """NVFP4 stack for one matrix kind; only `experts` are generated (others zero)."""
    return seeded.stack(spec, kind, experts, gen_device)


def oracle_layer(orc, spec: synth.LayerSpec, experts=None, gen_device="cpu"):
    """Oracle-side layer built from the same seeded bf16 tensors as the device layer."""
    return seeded.layer(spec, experts, gen_device)


def router_only_layer(orc, spec: synth.LayerSpec):
    """A layer whose expert stacks are empty placeholders: enough for orc.router."""
    return seeded.router_only_layer(spec)


def oracle_routes(orc, spec, x_bits: np.ndarray):
    """(logits [T, E], idx [T, k], w [T, k]) from the oracle router."""
    return seeded.routes(spec, x_bits)


def float_errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = got - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(err) / nref if nref > 0 else np.linalg.norm(err)
    rms = np.sqrt(np.mean(ref ** 2))
    mx = np.abs(err).max() if err.size else 0.0
    return rel, mx, rms


def assert_close(got, ref, what=""):
    rel, mx, rms = float_errors(got, ref)
    assert rel <= REL_L2, "%s: relative L2 %.3g > %.3g" % (what, rel, REL_L2)
    assert mx <= MAX_ABS_FRAC * rms, "%s: max abs %.3g > %.3g * rms %.3g" % (
        what, mx, MAX_ABS_FRAC, rms)
    return rel, mx


def routing_exempt(logits_row: np.ndarray, k: int) -> tuple[bool, bool]:
    """(set_exempt, order_exempt) for one token from the oracle's logits."""
    srt = np.sort(logits_row)[::-1]
    set_ex = k < len(srt) and (srt[k - 1] - srt[k]) < TIE_GAP
    order_ex = bool(np.any(np.diff(srt[:k]) > -TIE_GAP)) if k > 1 else False
    return set_ex, order_ex


def check_routing(gpu_idx, gpu_w, orc_logits, orc_idx, orc_w, k):
    """Asserts routing parity; returns a mask of tokens whose set matched exactly (the
    ones whose outputs are compared element by element)."""
    T = orc_idx.shape[0]
    ok = np.ones(T, bool)
    for t in range(T):
        set_ex, order_ex = routing_exempt(orc_logits[t], k)
        same_set = set(gpu_idx[t].tolist()) == set(orc_idx[t].tolist())
        if set_ex:
            ok[t] = same_set
            continue
        assert same_set, "token %d: expert set %s != oracle %s" % (t, gpu_idx[t], orc_idx[t])
        if not order_ex:
            np.testing.assert_array_equal(gpu_idx[t], orc_idx[t])
        # weights, matched by expert id
        wmap = dict(zip(orc_idx[t].tolist(), orc_w[t].tolist()))
        ref = np.array([wmap[int(e)] for e in gpu_idx[t]])
        assert_close(gpu_w[t], ref, "router weights token %d" % t)
    return ok
