"""GPU parity of the prompt-processing path (flint_moe_prefill) against the oracle's
prefill mode (activations NVFP4-quantised with unit tensor scale before each product).

Integer outputs (per-expert counts, the expert-major pair order) are bit-exact against
a plain counting sort of the GPU's own routing; the routing itself matches the oracle's
except near-ties; floats within relative L2 2e-3 and max-abs 1e-2 x RMS."""
import numpy as np
import pytest
import torch

from helpers import (assert_close, bits16, check_routing, oracle_layer, oracle_routes,
                     routing_exempt)
from sparse_moe_decode_02_b300 import flint, synth, workload

pytestmark = pytest.mark.gpu
DEV = "cuda"

MID = synth.MoeShape(hidden=512, n_experts=32, top_k=4, expert_width=256, shared_width=256,
                     vocab=4096)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flint.lib()


def _prefill(layer, x, E, k):
    T = x.shape[0]
    out = torch.empty(T, x.shape[1], dtype=torch.float32, device=DEV)
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    order = torch.empty(T * k, dtype=torch.int32, device=DEV)
    flint.moe_prefill(layer, x, out=out, topk_idx=idx, topk_w=w, expert_counts=counts,
                      pair_order=order)
    torch.cuda.synchronize()
    assert flint.last_device_status() == 0
    return (out.cpu().numpy().astype(np.float64), idx.cpu().numpy(), w.cpu().numpy(),
            counts.cpu().numpy(), order.cpu().numpy())


def _check_bookkeeping(orc, gidx, counts, order, E):
    ocounts, _, operm = orc.expert_order(gidx, E)
    np.testing.assert_array_equal(counts, ocounts)
    np.testing.assert_array_equal(order, operm)


@pytest.mark.parametrize("T,zipf,score", [(300, None, 0), (1, None, 0), (257, 1.1, 0),
                                          (200, 1.1, 1)])
def test_prefill_mid_all_tokens(orc, T, zipf, score):
    # score 1: the sigmoid router scoring (FLINT_ROUTER_SIGMOID)
    spec = synth.LayerSpec(MID, seed=31, zipf=zipf, router_score=score)
    layer = workload.build_layer(spec, DEV)
    x = synth.tokens_bf16(31, MID.hidden, T, stream=7)
    out, gidx, gw, counts, order = _prefill(layer, x.to(DEV), MID.n_experts, MID.top_k)
    xb = bits16(x)
    logits, oidx, ow = oracle_routes(orc, spec, xb)
    ok = check_routing(gidx, gw, logits, oidx, ow, MID.top_k)
    _check_bookkeeping(orc, gidx, counts, order, MID.n_experts)
    L = oracle_layer(orc, spec)
    oout, _, _ = orc.moe_forward(L, xb, quantize_acts=True)
    xd = x.double().numpy()
    assert_close(out[ok] - xd[ok], oout[ok] - xd[ok], "prefill MoE delta")
    assert_close(out[ok], oout[ok], "prefill out")


def test_prefill_flint_config(orc):
    """The Flint prompt-processing layer: 4096 tokens, 256 experts top-6 with a Zipf(1.1)
    router bias, shared expert 1024.  Routing, counts and order on every token; the
    outputs of the first and the last token of every 128-row tile of every expert's
    token list (where the grouped GEMM masks a partial tile) and of every tile of the
    shared expert, against the oracle."""
    shape = synth.FLINT
    T, E, k = 4096, shape.n_experts, shape.top_k
    spec = synth.LayerSpec(shape, seed=0, zipf=1.1)
    layer = workload.build_layer(spec, DEV)
    x = synth.tokens_bf16(0, shape.hidden, T, stream=9)
    out, gidx, gw, counts, order = _prefill(layer, x.to(DEV), E, k)
    xb = bits16(x)
    logits, oidx, ow = oracle_routes(orc, spec, xb)
    ok = check_routing(gidx, gw, logits, oidx, ow, k)
    _check_bookkeeping(orc, gidx, counts, order, E)
    offs = np.concatenate([[0], np.cumsum(counts)[:-1]])
    pick = set()
    for e in range(E):
        for r0 in range(0, int(counts[e]), 128):
            r1 = min(r0 + 127, int(counts[e]) - 1)
            pick.add(int(order[offs[e] + r0]) // k)
            pick.add(int(order[offs[e] + r1]) // k)
    for r0 in range(0, T, 128):
        pick.update((r0, min(r0 + 127, T - 1)))
    sample = np.array(sorted(pick))
    tiles = sum((int(c) + 127) // 128 for c in counts)
    sample = sample[ok[sample]]
    assert len(sample) >= tiles // 2
    L = oracle_layer(orc, spec, experts=np.unique(oidx[sample]), gen_device=DEV)
    oout, _, _ = orc.moe_forward(L, xb[sample], quantize_acts=True)
    xd = x.double().numpy()[sample]
    for i, t in enumerate(sample):
        assert_close(out[t] - xd[i], oout[i] - xd[i], "prefill MoE delta, token %d" % t)
    # and close to the unquantised layer (the activation quantisation error only)
    plain, _, _ = orc.moe_forward(L, xb[sample])
    rel = np.linalg.norm((out[sample] - xd) - (plain - xd)) / np.linalg.norm(plain - xd)
    assert rel < 0.2


def test_prefill_matches_decode_routing():
    """The prefill router (tensor-core bf16 GEMM) and the decode router (bf16 GEMV) pick
    the same experts for the same tokens (outside near-ties)."""
    spec = synth.LayerSpec(MID, seed=33)
    layer = workload.build_layer(spec, DEV)
    x = synth.tokens_bf16(33, MID.hidden, 40, stream=8).to(DEV)
    _, pidx, pw, _, _ = _prefill(layer, x, MID.n_experts, MID.top_k)
    didx = torch.empty(40, MID.top_k, dtype=torch.int32, device=DEV)
    dw = torch.empty(40, MID.top_k, dtype=torch.float32, device=DEV)
    for t0 in range(0, 40, 8):
        flint.moe_decode(layer, x[t0:t0 + 8], topk_idx=didx[t0:t0 + 8], topk_w=dw[t0:t0 + 8])
    torch.cuda.synchronize()
    same = (np.sort(pidx, 1) == np.sort(didx.cpu().numpy(), 1)).all(1)
    assert same.mean() >= 0.95
