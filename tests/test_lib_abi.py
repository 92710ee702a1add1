"""CPU checks of the C-ABI library: it loads, exports every function include/flint.h
declares, and rejects bad arguments on the host before anything is enqueued (these
calls never reach the GPU, so they run without one)."""
import ctypes
import os
import re

import pytest

from sparse_moe_decode_02_b300 import build, flint

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flint.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return flint.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flint_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_north_star_calls():
    names = declared_functions()
    for n in ("flint_quantize_nvfp4", "flint_moe_decode", "flint_moe_prefill", "flint_lm_head"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_host_only_helpers(L):
    assert b"sm_103a" in L.flint_version()
    for s in range(9):
        assert len(L.flint_status_string(s)) > 0
    nb = flint.workspace_bytes(flint.OP_MOE_DECODE, 2048, 256, 6, 512, 1024, 0, 1)
    assert nb > 0 and nb % 256 == 0
    assert flint.workspace_bytes(flint.OP_LM_HEAD, 2048, 0, 0, 0, 0, 150144, 8) > 0
    assert flint.workspace_bytes(flint.OP_MOE_PREFILL, 2048, 256, 6, 512, 1024, 0, 4096) > 0


FAKE = 0x10000000        # aligned, never dereferenced: the checks fail first
FAKE_MIS = 0x10000008    # 8-byte aligned only


def _nv(n, r, c, codes=FAKE):
    return flint._NVFP4C(codes, FAKE, FAKE, n, r, c)


def _layer(H=256, E=16, k=2, F=64, Fs=128, router=FAKE, gate_cols=None, sf=FAKE, score=0):
    return flint._LayerC(H, E, k, F, Fs, router, None, _nv(E, F, gate_cols or H), _nv(E, F, H),
                         _nv(E, H, F), _nv(1, Fs, H), _nv(1, Fs, H), _nv(1, H, Fs),
                         (ctypes.c_void_p * 6)(*[sf] * 6), score)


def test_quantize_argument_checks(L):
    q = L.flint_quantize_nvfp4
    assert q(None, 1, 8, 32, FAKE, FAKE, FAKE, FAKE, 256, None) == 1
    assert q(FAKE, 1, 8, 48, FAKE, FAKE, FAKE, FAKE, 256, None) == 3       # cols % 32
    assert q(FAKE, 0, 8, 32, FAKE, FAKE, FAKE, FAKE, 256, None) == 1
    assert q(FAKE_MIS, 1, 8, 32, FAKE, FAKE, FAKE, FAKE, 256, None) == 2
    assert q(FAKE, 1, 8, 32, FAKE, FAKE, FAKE, FAKE + 16, 256, None) == 4  # ws alignment
    assert q(FAKE, 1000, 8, 32, FAKE, FAKE, FAKE, FAKE, 256, None) == 4    # ws size


def test_decode_argument_checks(L):
    d = L.flint_moe_decode
    lay = _layer()
    ws = flint.workspace_bytes(flint.OP_MOE_DECODE, 256, 16, 2, 64, 128, 0, 1)
    args = lambda **kw: dict(dict(x=FAKE, res=None, out=FAKE, xn=None, eps=1e-6, idx=None,
                                  w=None, B=1, ws=FAKE, wsb=ws), **kw)
    call = lambda lay, a: d(ctypes.byref(lay), a["x"], a["res"], a["out"], a["xn"], a["eps"],
                            a["idx"], a["w"], a["B"], a["ws"], a["wsb"], None)
    assert d(None, FAKE, None, FAKE, None, 1e-6, None, None, 1, FAKE, ws, None) == 1
    assert call(lay, args(B=0)) == 1
    assert call(lay, args(B=9)) == 8                                    # > FLINT_MAX_DECODE_TOKENS
    assert call(lay, args(x=FAKE_MIS)) == 2
    assert call(lay, args(wsb=ws - 1)) == 4
    assert call(_layer(k=17, E=32), args()) == 8                        # top_k > MAX
    assert call(_layer(k=20, E=16), args()) == 1                        # k > E
    assert call(_layer(H=96), args()) == 8                              # not a power of two
    assert call(_layer(H=250), args()) == 3                             # not a multiple of 32
    assert call(_layer(gate_cols=512), args()) == 3                     # stack shape mismatch
    assert call(_layer(router=FAKE_MIS), args()) == 2
    assert call(_layer(score=2), args()) == 1                           # unknown router scoring
    assert call(_layer(score=-1), args()) == 1


def test_decode_tokens_argument_checks(L):
    dt = L.flint_decode_tokens
    ws = flint.workspace_bytes(flint.OP_MOE_DECODE, 256, 16, 2, 64, 128, 0, 4)
    arr = (flint._LayerC * 3)(_layer(), _layer(), _layer())
    head = _nv(1, 4096, 256)
    ok = lambda **kw: dict(dict(layers=arr, n=3, head=ctypes.byref(head), x=FAKE, res=None, T=4,
                                eps=1e-6, out=None, xo=None, lg=None, am=FAKE, ti=None, tw=None,
                                ws=FAKE, wsb=ws), **kw)
    call = lambda a: dt(a["layers"], a["n"], a["head"], a["x"], a["res"], a["T"], a["eps"],
                        a["out"], a["xo"], a["lg"], a["am"], a["ti"], a["tw"], a["ws"], a["wsb"],
                        None)
    assert call(ok(n=0)) == 1
    assert call(ok(n=65)) == 8                                          # > FLINT_MAX_LAYERS
    assert call(ok(T=0)) == 1
    assert call(ok(head=None)) == 1                                     # argmax without a head
    bad_head = _nv(1, 4096, 512)
    assert call(ok(head=ctypes.byref(bad_head))) == 3                   # head cols != hidden
    mixed = (flint._LayerC * 2)(_layer(), _layer(H=512))
    assert call(ok(layers=mixed, n=2)) == 3                             # layers of unequal hidden
    assert call(ok(eps=-1.0)) == 1
    assert call(ok(wsb=16)) == 4


def test_decode_trace_and_wait_controls(L):
    tr = L.flint_decode_tokens_trace
    ws = flint.workspace_bytes(flint.OP_MOE_DECODE, 256, 16, 2, 64, 128, 0, 4)
    arr = (flint._LayerC * 1)(_layer())
    call = lambda xt, ht: tr(arr, 1, None, FAKE, None, 2, 1e-6, FAKE, None, None, None, None,
                             None, xt, ht, FAKE, ws, None)
    assert call(FAKE_MIS, None) == 2                                   # trace rows 16-byte aligned
    assert call(None, FAKE + 4) == 2
    assert L.flint_set_wait_limit_ns(5_000_000) == 0
    assert L.flint_set_wait_limit_ns(0) == 0                           # back to the default
    assert L.flint_debug_hold_next_launch(3) == 1
    assert L.flint_debug_hold_next_launch(-1) == 1
    assert L.flint_debug_hold_next_launch(0) == 0


def test_mma_scales_argument_checks(L):
    ms = L.flint_nvfp4_mma_scales
    assert ms(None, FAKE, None) == 1
    assert ms(ctypes.byref(_nv(2, 128, 256)), None, None) == 1
    assert ms(ctypes.byref(_nv(2, 64, 256)), FAKE, None) == 3             # rows % 128
    assert ms(ctypes.byref(_nv(2, 128, 96)), FAKE, None) == 3             # cols % 64
    assert ms(ctypes.byref(_nv(2, 128, 256)), FAKE_MIS, None) == 2


def test_prefill_argument_checks(L):
    p = L.flint_moe_prefill
    H, E, k, F, Fs, T = 512, 32, 4, 256, 256, 64
    ws = flint.workspace_bytes(flint.OP_MOE_PREFILL, H, E, k, F, Fs, 0, T)
    good = _layer(H, E, k, F, Fs)
    assert p(None, FAKE, FAKE, None, None, None, None, T, FAKE, ws, None) == 1
    assert p(ctypes.byref(good), FAKE, FAKE, None, None, None, None, 0, FAKE, ws, None) == 1
    assert p(ctypes.byref(_layer(H, E, k, F, Fs, sf=0)), FAKE, FAKE, None, None, None, None, T,
             FAKE, ws, None) == 1                                          # no MMA scale copies
    assert p(ctypes.byref(_layer(H, E, k, F, Fs, sf=FAKE_MIS)), FAKE, FAKE, None, None, None,
             None, T, FAKE, ws, None) == 2
    assert p(ctypes.byref(_layer(256, 16, 2, 64, 128)), FAKE, FAKE, None, None, None, None, T,
             FAKE, ws, None) == 8                                          # F % 256
    assert p(ctypes.byref(good), FAKE, FAKE, None, None, None, None, T, FAKE, 16, None) == 4


def test_lm_head_argument_checks(L):
    h = L.flint_lm_head
    W = _nv(1, 4096, 256)
    ws = flint.workspace_bytes(flint.OP_LM_HEAD, 256, 0, 0, 0, 0, 4096, 1)
    assert h(ctypes.byref(W), FAKE, None, None, 1, FAKE, ws, None) == 1   # no output at all
    assert h(ctypes.byref(W), FAKE, FAKE, None, 0, FAKE, ws, None) == 1
    assert h(ctypes.byref(W), FAKE, FAKE, None, 9, FAKE, ws, None) == 8
    W2 = _nv(2, 4096, 256)
    assert h(ctypes.byref(W2), FAKE, FAKE, None, 1, FAKE, ws, None) == 3
    assert h(ctypes.byref(W), FAKE_MIS, FAKE, None, 1, FAKE, ws, None) == 2
    assert h(ctypes.byref(W), FAKE, FAKE, None, 1, FAKE, 16, None) == 4


def test_sample_argument_checks(L):
    s = L.flint_sample_logits
    ok = dict(lg=FAKE, B=2, V=100, T=1.0, k=20, p=0.95, u=FAKE, out=FAKE)
    call = lambda **kw: s(*(dict(ok, **kw)[n] for n in ("lg", "B", "V", "T", "k", "p", "u", "out")), None)
    assert call(lg=None) == 1
    assert call(u=None) == 1
    assert call(out=None) == 1
    assert call(B=0) == 1
    assert call(V=0) == 1
    assert call(k=0) == 1
    assert call(k=33) == 8                                               # > FLINT_MAX_SAMPLE_TOP_K
    assert call(T=0.0) == 1
    assert call(T=float("inf")) == 1
    assert call(p=0.0) == 1
    assert call(p=1.5) == 1
    assert call(lg=FAKE + 2) == 2


def test_decode_tokens_sample_argument_checks(L):
    ds = L.flint_decode_tokens_sample
    ws = flint.workspace_bytes(flint.OP_MOE_DECODE, 256, 16, 2, 64, 128, 0, 4)
    arr = (flint._LayerC * 1)(_layer())
    head = _nv(1, 4096, 256)
    ok = dict(head=ctypes.byref(head), temp=1.0, k=20, p=0.95, u=FAKE, tok=FAKE)
    call = lambda **kw: ds(arr, 1, dict(ok, **kw)["head"], FAKE, None, 2, 1e-6, dict(ok, **kw)["temp"],
                           dict(ok, **kw)["k"], dict(ok, **kw)["p"], dict(ok, **kw)["u"],
                           dict(ok, **kw)["tok"], None, None, None, None, None, None, FAKE, ws, None)
    assert call(head=None) == 1
    assert call(u=None) == 1
    assert call(tok=None) == 1
    assert call(temp=0.0) == 1
    assert call(temp=float("inf")) == 1
    assert call(p=0.0) == 1
    assert call(p=1.5) == 1
    assert call(k=0) == 1
    assert call(k=33) == 8                                               # > FLINT_MAX_SAMPLE_TOP_K
    assert call(tok=FAKE + 2) == 2


def test_dense_layer_checks(L):
    # a dense SwiGLU layer: n_experts = top_k = expert_width = 0, the block in sh_*
    dense = flint._LayerC(256, 0, 0, 0, 384, None, None, _nv(0, 0, 256), _nv(0, 0, 256),
                          _nv(0, 256, 0), _nv(1, 384, 256), _nv(1, 384, 256), _nv(1, 256, 384),
                          (ctypes.c_void_p * 6)(*[None] * 6), 0)
    ws = flint.workspace_bytes(flint.OP_MOE_DECODE, 256, 0, 0, 0, 384, 0, 1)
    d = L.flint_moe_decode
    # the checks accept it; with no GPU here the call then stops at the device query
    assert d(ctypes.byref(dense), FAKE, None, FAKE, None, 1e-6, None, None, 1, FAKE, ws, None) == 7
    bad = flint._LayerC(256, 0, 0, 0, 200, None, None, _nv(0, 0, 256), _nv(0, 0, 256),
                        _nv(0, 256, 0), _nv(1, 200, 256), _nv(1, 200, 256), _nv(1, 256, 200),
                        (ctypes.c_void_p * 6)(*[None] * 6), 0)
    assert d(ctypes.byref(bad), FAKE, None, FAKE, None, 1e-6, None, None, 1, FAKE, ws, None) == 3
    p = L.flint_moe_prefill
    assert p(ctypes.byref(dense), FAKE, FAKE, None, None, None, None, 4, FAKE, 1 << 30, None) == 8
