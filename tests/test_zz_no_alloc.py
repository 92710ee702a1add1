"""The no-allocation decode entry point (flint_decode_tokens_noalloc) against the
workspace one (flint_decode_tokens).

flint_decode_tokens_noalloc serves callers that cannot allocate device scratch -- a
host that owns all device memory and gives extensions no allocator, or a serving loop
that must not call cudaMalloc.  It keeps its scratch in a fixed device array inside the
library.  This file is collected last on purpose: run after the other tests, it also
checks that the shared array's leftover contents from earlier calls do no harm.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close, TIE_GAP
from sparse_moe_decode_02_b300 import flint, synth, workload

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(fn, layers, head, x, shape, T, L):
    H, k, V = shape.hidden, shape.top_k, shape.vocab
    res = dict(out=torch.empty(T, H, dtype=torch.float32, device=DEV),
               x_out=torch.empty(T, H, dtype=torch.bfloat16, device=DEV),
               logits=torch.empty(T, V, dtype=torch.float32, device=DEV),
               argmax=torch.empty(T, dtype=torch.int32, device=DEV),
               topk_idx=torch.empty(T, L, k, dtype=torch.int32, device=DEV),
               topk_w=torch.empty(T, L, k, dtype=torch.float32, device=DEV))
    fn(layers, x, head=head, rms_eps=1e-6, **res)
    torch.cuda.synchronize()
    return {n: t.cpu() for n, t in res.items()}


# a hidden size below the widest and the most experts the decode accepts, with more selected
# experts than routed clusters (so some clusters run two routed passes)
WIDE = synth.MoeShape(hidden=1024, n_experts=256, top_k=8, expert_width=256, shared_width=512,
                      vocab=4096)


@pytest.mark.parametrize("shape,L,T", [(synth.TINY, 3, 5), (synth.FLINT, 2, 3), (WIDE, 1, 2)])
def test_noalloc_matches_workspace_entry_point_twice(shape, L, T):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    flint.lib()
    layers = [workload.build_layer(synth.LayerSpec(shape, seed=21, layer=l, zipf=1.1), DEV)
              for l in range(L)]
    head = workload.build_head(21, shape.vocab, shape.hidden, DEV)
    x = synth.tokens_bf16(21, shape.hidden, T, stream=5).to(DEV)
    ref = _run(flint.decode_tokens, layers, head, x, shape, T, L)
    assert flint.last_device_status() == 0
    for call in range(2):          # two calls in a row share the fixed scratch
        got = _run(flint.decode_tokens_noalloc, layers, head, x, shape, T, L)
        assert flint.last_device_status() == 0
        assert_close(got["out"].double().numpy(), ref["out"].double().numpy(), "out, call %d" % call)
        assert_close(got["logits"].double().numpy(), ref["logits"].double().numpy(),
                     "logits, call %d" % call)
        assert_close(got["topk_w"].double().numpy(), ref["topk_w"].double().numpy(),
                     "router weights, call %d" % call)
        np.testing.assert_array_equal(np.sort(got["topk_idx"].numpy(), -1),
                                      np.sort(ref["topk_idx"].numpy(), -1))
        d = (got["x_out"].float() - ref["x_out"].float()).abs().max().item()
        assert d <= 2.0 ** -6 * ref["x_out"].float().abs().max().item()
        lg = ref["logits"].numpy()
        for t in range(T):
            srt = np.sort(lg[t])[::-1]
            if srt[0] - srt[1] >= TIE_GAP:
                assert int(got["argmax"][t]) == int(ref["argmax"][t])


def test_noalloc_scratch_covers_every_supported_shape():
    # the scratch depends on the hidden size only; the widest one accepted (2048) fits
    flint.lib()
    full = flint.workspace_bytes(flint.OP_MOE_DECODE, 2048, 256, 6, 512, 1024, 0, 1)
    assert full <= 512 * 1024
