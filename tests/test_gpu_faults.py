"""Bounded device waits run out without a fault: a launch armed with
flint_debug_hold_next_launch withholds one hand-over, its waits expire after a short
flint_set_wait_limit_ns, the device status reads FLINT_ERR_TIMEOUT, and the next normal
call on the same context succeeds with the results of an undisturbed run.  No GPU fault,
trap or endless wait is involved: every wait is bounded and the kernel unwinds."""
import numpy as np
import pytest
import torch

from helpers import assert_close
from sparse_moe_decode_02_b300 import flint, synth, workload

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT = 6          # FLINT_ERR_TIMEOUT
SHORT_NS = 20_000_000


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flint.lib()
    yield
    flint.set_wait_limit_ns(0)
    flint.debug_hold_next_launch(0)


def _decode(layers, head, x, shape, L):
    T, H = x.shape
    res = dict(out=torch.empty(T, H, dtype=torch.float32, device=DEV),
               logits=torch.empty(T, shape.vocab, dtype=torch.float32, device=DEV),
               argmax=torch.empty(T, dtype=torch.int32, device=DEV),
               topk_idx=torch.empty(T, L, shape.top_k, dtype=torch.int32, device=DEV))
    flint.decode_tokens(layers, x, head=head, **res)
    status = flint.last_device_status()            # synchronises
    return status, {n: t.cpu() for n, t in res.items()}


def test_decode_wait_expires_then_next_call_is_good():
    shape, L = synth.TINY, 3
    layers = [workload.build_layer(synth.LayerSpec(shape, seed=41, layer=l, zipf=1.1), DEV)
              for l in range(L)]
    head = workload.build_head(41, shape.vocab, shape.hidden, DEV)
    x = synth.tokens_bf16(41, shape.hidden, 3, stream=2).to(DEV)
    st, ref = _decode(layers, head, x, shape, L)
    assert st == 0
    flint.set_wait_limit_ns(SHORT_NS)
    flint.debug_hold_next_launch(1)
    st, _ = _decode(layers, head, x, shape, L)
    assert st == TIMEOUT
    flint.set_wait_limit_ns(0)
    st, got = _decode(layers, head, x, shape, L)
    assert st == 0
    for n in ref:                                  # the decode is deterministic
        assert torch.equal(got[n], ref[n]), n


def test_prefill_wait_expires_then_next_call_is_good():
    shape = synth.MoeShape(hidden=512, n_experts=32, top_k=4, expert_width=256,
                           shared_width=256)
    layer = workload.build_layer(synth.LayerSpec(shape, seed=42, zipf=1.1), DEV)
    x = synth.tokens_bf16(42, shape.hidden, 300, stream=3).to(DEV)

    def run():
        out = flint.moe_prefill(layer, x)
        return flint.last_device_status(), out.cpu().numpy().astype(np.float64)

    st, ref = run()
    assert st == 0
    flint.set_wait_limit_ns(SHORT_NS)
    flint.debug_hold_next_launch(2)
    st, _ = run()
    assert st == TIMEOUT
    flint.set_wait_limit_ns(0)
    st, got = run()
    assert st == 0
    assert_close(got, ref, "prefill after an expired wait")
