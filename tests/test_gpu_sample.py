"""Sampling after the output head (flint_sample_logits) against the oracle: the drawn
index per row, exact except where the caller's uniform or top_p lies within float
rounding of a cumulative sum (the kernel sums in fp32, the oracle in fp64)."""
import numpy as np
import pytest
import torch
from scipy.special import softmax

from sparse_moe_decode_02_b300 import flint

pytestmark = pytest.mark.gpu
DEV = "cuda"
NEAR = 1e-5


def _near_boundary(row, T, k, top_p, u):
    """True when the fp64 decision points lie within NEAR of top_p or of u."""
    r = np.where(np.isnan(row), -np.inf, row.astype(np.float64))
    k = min(k, r.size)
    order = np.argsort(-r, kind="stable")[:k]
    if np.isinf(r[order[0]]):          # all -inf, or a +inf logit: no sums decide
        return False
    c = np.cumsum(softmax((r[order] - r[order[0]]) / T))
    # the last sum decides nothing: m = k whether or not it reaches top_p
    if k > 1 and np.min(np.abs(c[:-1] - top_p)) < NEAR:
        return True
    m = int(np.argmax(c >= top_p)) + 1 if np.any(c >= top_p) else k
    cq = c[:m] / c[m - 1]
    return bool(np.min(np.abs(cq - u)) < NEAR)


def _check(orc, logits, uniforms, T, k, top_p):
    """Compares every row not near a boundary; returns the number of rows skipped."""
    got = flint.sample_logits(torch.from_numpy(logits).to(DEV), torch.from_numpy(uniforms),
                              temperature=T, top_k=k, top_p=top_p).cpu().numpy()
    torch.cuda.synchronize()
    skipped = 0
    for b in range(logits.shape[0]):
        if _near_boundary(logits[b], T, k, top_p, float(uniforms[b])):
            skipped += 1
            continue
        want, _ = orc.sample(logits[b], T, k, top_p, float(uniforms[b]))
        assert got[b] == want, (b, got[b], want)
    return skipped


@pytest.mark.parametrize("T,k,top_p", [(1.0, 20, 0.95), (0.7, 32, 0.5), (1.0, 1, 0.95),
                                       (2.0, 20, 1.0)])
def test_sample_head_vocab(orc, T, k, top_p):
    # 16 rows over the Flint vocabulary (150,144), logits N(0, 3^2)
    rng = np.random.default_rng(int(T * 10) + k)
    logits = (rng.standard_normal((16, 150144)) * 3).astype(np.float32)
    uniforms = rng.random(16).astype(np.float32)
    assert _check(orc, logits, uniforms, T, k, top_p) <= 4


def test_sample_ties_nan_and_small_vocab(orc):
    rng = np.random.default_rng(7)
    cases = [(np.round(rng.standard_normal(3001)).astype(np.float32), 20, 0.95),   # many ties
             (np.full(500, 0.25, np.float32), 16, 0.95),                          # all equal
             (np.full(500, 0.25, np.float32), 16, 0.4),
             ((rng.standard_normal(1000) * 2).astype(np.float32), 20, 0.95),
             (np.array([1.0, -2.0, 0.5, 3.0, 0.0], np.float32), 20, 0.95),       # V < top_k
             (np.full(64, -np.inf, np.float32), 20, 0.95),                        # all -inf
             (np.array([0.5, np.inf, 3.0, np.inf, -1.0] * 40, np.float32), 20, 0.95)]  # +inf
    cases[3][0][rng.integers(0, 1000, 100)] = np.nan
    checked = skipped = 0
    for row, k, top_p in cases:
        for u in (0.0, 0.37, 0.91):
            skipped += _check(orc, row[None].copy(), np.array([u], np.float32), 1.0, k, top_p)
            checked += 1
    assert skipped <= checked // 4


@pytest.mark.parametrize("shape_name,L,T,temp,k,top_p", [("FLINT", 2, 6, 1.0, 20, 0.95),
                                                          ("FLINT", 1, 4, 0.6, 32, 0.8),
                                                          ("TINY", 3, 8, 1.0, 20, 0.95),
                                                          ("TINY", 2, 5, 1.5, 1, 0.95)])
def test_decode_fused_sampling(orc, shape_name, L, T, temp, k, top_p):
    """flint_decode_tokens_sample: the token drawn inside the decode launch equals the
    oracle's draw from the same logits (the launch also writes them), the argmax is the
    first candidate, and the rest of the launch matches flint_decode_tokens."""
    from sparse_moe_decode_02_b300 import synth, workload
    shape = getattr(synth, shape_name)
    layers = [workload.build_layer(synth.LayerSpec(shape, seed=51, layer=l, zipf=1.1), DEV)
              for l in range(L)]
    head = workload.build_head(51, shape.vocab, shape.hidden, DEV)
    x = synth.tokens_bf16(51, shape.hidden, T, stream=6).to(DEV)
    rng = np.random.default_rng(T + k)
    u = torch.from_numpy(rng.random(T).astype(np.float32)).to(DEV)
    lg = torch.empty(T, shape.vocab, dtype=torch.float32, device=DEV)
    am = torch.empty(T, dtype=torch.int32, device=DEV)
    out = torch.empty(T, shape.hidden, dtype=torch.float32, device=DEV)
    tok = flint.decode_tokens_sample(layers, x, head, u, temperature=temp, top_k=k, top_p=top_p,
                                     logits=lg, argmax=am, out=out)
    torch.cuda.synchronize()
    assert flint.last_device_status() == 0
    lg2 = torch.empty_like(lg)
    out2 = torch.empty_like(out)
    flint.decode_tokens(layers, x, head=head, logits=lg2, out=out2)
    torch.cuda.synchronize()
    assert torch.equal(lg, lg2) and torch.equal(out, out2)
    logits, tok, am, u = lg.cpu().numpy(), tok.cpu().numpy(), am.cpu().numpy(), u.cpu().numpy()
    skipped = 0
    for t in range(T):
        assert am[t] == int(np.argmax(logits[t]))
        if _near_boundary(logits[t], temp, k, top_p, float(u[t])):
            skipped += 1
            continue
        want, _ = orc.sample(logits[t], temp, k, top_p, float(u[t]))
        assert tok[t] == want, (t, tok[t], want)
    assert skipped <= T // 2
