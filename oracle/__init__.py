"""Plain CPU oracle for the Flint NVFP4 MoE feed-forward and output head.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The library's product path never loads it, and it imports nothing from
the library: the two share no code.  The arithmetic lives in ``flint_oracle.c``
(C, fp64; the quantiser in fp32 where the bytes are defined); this module only
marshals numpy arrays through ctypes.

Page citations and the readings taken where the pages are silent are in
``flint_oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "flint_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-ffp-contract=off: fp32 steps stay IEEE)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(_SRC[:-2] + ".h"))):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O3", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fno-fast-math", "-pthread", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _NVFP4(ctypes.Structure):
    _fields_ = [("codes", _u8p), ("scales", _u8p), ("tsc", _f32p)]


class _Layer(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("expert_width", ctypes.c_int),
                ("shared_width", ctypes.c_int),
                ("router_w", _u16p), ("router_bias", _f32p),
                ("gate", _NVFP4), ("up", _NVFP4), ("down", _NVFP4),
                ("sh_gate", _NVFP4), ("sh_up", _NVFP4), ("sh_down", _NVFP4),
                ("router_score", ctypes.c_int)]

ROUTER_SOFTMAX, ROUTER_SIGMOID = 0, 1


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        L = _lib
        L.orc_e2m1_value.restype = ctypes.c_double
        L.orc_e4m3_value.restype = ctypes.c_double
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e2m1_encode.restype = ctypes.c_uint8
        L.orc_e2m1_encode.argtypes = [ctypes.c_float]
        L.orc_bf16_value.restype = ctypes.c_double
        L.orc_bf16_value.argtypes = [ctypes.c_uint16]
        L.orc_bf16_from_double.restype = ctypes.c_uint16
        L.orc_bf16_from_double.argtypes = [ctypes.c_double]
        L.orc_quantize_nvfp4.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _u8p, _f32p]
        L.orc_quantize_rows_unit.argtypes = [_f32p, _i64, _i64, _u8p, _u8p]
        L.orc_dequantize_nvfp4.argtypes = [_u8p, _u8p, _f32p, _i64, _i64, _i64, _f32p]
        L.orc_router.argtypes = [ctypes.POINTER(_Layer), _u16p, _f64p, _i32p, _f64p]
        L.orc_sample.argtypes = [_f32p, ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                 ctypes.c_double, ctypes.c_double, ctypes.POINTER(ctypes.c_int)]
        L.orc_sample.restype = ctypes.c_int32
        L.orc_moe_forward.argtypes = [ctypes.POINTER(_Layer), _u16p, _f64p, _i64,
                                      ctypes.c_int, _f64p, _i32p, _f64p]
        L.orc_rmsnorm_bf16.argtypes = [_f64p, _i64, ctypes.c_double, _u16p]
        L.orc_lm_head.argtypes = [ctypes.POINTER(_NVFP4), _i64, _i64, _u16p, _i64,
                                  _f64p, _i32p]
        L.orc_expert_order.argtypes = [_i32p, _i64, ctypes.c_int, ctypes.c_int,
                                       _i32p, _i32p, _i32p]
        L.orc_set_threads(os.cpu_count() or 1)
    return _lib


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


def _p(a, t):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(t)


def _bits16(a):
    """bf16 data as uint16 bits (accepts uint16 arrays or torch bf16 tensors)."""
    if hasattr(a, "view") and str(getattr(a, "dtype", "")) == "torch.bfloat16":
        import torch
        return a.contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


# --------------------------------------------------------------------------- formats
def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def e4m3_value(byte: int) -> float:
    return lib().orc_e4m3_value(int(byte))


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def e2m1_encode(v: float) -> int:
    return int(lib().orc_e2m1_encode(float(v)))


def bf16_from_double(v: float) -> int:
    return int(lib().orc_bf16_from_double(float(v)))


# --------------------------------------------------------------------------- quantiser
class NVFP4:
    """An oracle-side NVFP4 stack: codes [n, R, C/2], scales [n, R, C/16], tsc [n]."""

    def __init__(self, codes, scales, tsc):
        self.codes = np.ascontiguousarray(codes, dtype=np.uint8)
        self.scales = np.ascontiguousarray(scales, dtype=np.uint8)
        self.tsc = np.ascontiguousarray(tsc, dtype=np.float32)

    @property
    def shape(self):
        n, r, half = self.codes.shape
        return n, r, half * 2

    def c(self):
        return _NVFP4(_p(self.codes, _u8p), _p(self.scales, _u8p), _p(self.tsc, _f32p))

    def dequantize(self) -> np.ndarray:
        n, r, c = self.shape
        out = np.empty((n, r, c), np.float32)
        lib().orc_dequantize_nvfp4(_p(self.codes, _u8p), _p(self.scales, _u8p),
                                   _p(self.tsc, _f32p), n, r, c, _p(out, _f32p))
        return out


def quantize_nvfp4(w_bf16) -> tuple[NVFP4, int]:
    """bf16 [n, R, C] (uint16 bits or torch bf16) -> (NVFP4, status)."""
    w = _bits16(w_bf16)
    if w.ndim == 2:
        w = w[None]
    n, r, c = w.shape
    codes = np.zeros((n, r, c // 2), np.uint8)
    scales = np.zeros((n, r, c // 16), np.uint8)
    tsc = np.zeros((n,), np.float32)
    st = lib().orc_quantize_nvfp4(_p(w, _u16p), n, r, c, _p(codes, _u8p), _p(scales, _u8p),
                                  _p(tsc, _f32p))
    return NVFP4(codes, scales, tsc), int(st)


def quantize_rows_unit(v: np.ndarray):
    """fp32 rows [R, C] -> codes [R, C/2], scales [R, C/16] with tensor scale 1."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    r, c = v.shape
    codes = np.zeros((r, c // 2), np.uint8)
    scales = np.zeros((r, c // 16), np.uint8)
    lib().orc_quantize_rows_unit(_p(v, _f32p), r, c, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


# --------------------------------------------------------------------------- MoE layer
class Layer:
    """Oracle-side MoE layer.  Matrices are NVFP4 stacks; router_w is bf16 bits."""

    def __init__(self, router_w, router_bias, gate, up, down, sh_gate, sh_up, sh_down, top_k,
                 router_score=ROUTER_SOFTMAX):
        self.router_w = _bits16(router_w)
        self.router_bias = (None if router_bias is None
                            else np.ascontiguousarray(router_bias, dtype=np.float32))
        self.gate, self.up, self.down = gate, up, down
        self.sh_gate, self.sh_up, self.sh_down = sh_gate, sh_up, sh_down
        self.top_k = int(top_k)
        self.router_score = int(router_score)
        self.n_experts, self.hidden = self.router_w.shape
        self.expert_width = gate.shape[1]
        self.shared_width = sh_gate.shape[1]

    def c(self):
        return _Layer(self.hidden, self.n_experts, self.top_k, self.expert_width,
                      self.shared_width, _p(self.router_w, _u16p),
                      _p(self.router_bias, _f32p), self.gate.c(), self.up.c(),
                      self.down.c(), self.sh_gate.c(), self.sh_up.c(), self.sh_down.c(),
                      self.router_score)


def router(layer: Layer, x_bf16):
    x = _bits16(x_bf16).reshape(-1)
    logits = np.zeros(layer.n_experts, np.float64)
    idx = np.zeros(layer.top_k, np.int32)
    w = np.zeros(layer.top_k, np.float64)
    cl = layer.c()
    lib().orc_router(ctypes.byref(cl), _p(x, _u16p), _p(logits, _f64p), _p(idx, _i32p),
                     _p(w, _f64p))
    return logits, idx, w


def moe_forward(layer: Layer, x_bf16, residual=None, quantize_acts=False):
    """x bf16 [T, H] -> (out fp64 [T, H], idx [T, k], w fp64 [T, k])."""
    x = _bits16(x_bf16)
    if x.ndim == 1:
        x = x[None]
    T, H = x.shape
    out = np.zeros((T, H), np.float64)
    idx = np.zeros((T, layer.top_k), np.int32)
    w = np.zeros((T, layer.top_k), np.float64)
    res = None if residual is None else np.ascontiguousarray(residual, dtype=np.float64)
    cl = layer.c()
    st = lib().orc_moe_forward(ctypes.byref(cl), _p(x, _u16p), _p(res, _f64p), T,
                               1 if quantize_acts else 0, _p(out, _f64p), _p(idx, _i32p),
                               _p(w, _f64p))
    if st != 0:
        raise ValueError("oracle moe_forward status %d" % st)
    return out, idx, w


def rmsnorm_bf16(h: np.ndarray, eps: float) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.float64).reshape(-1)
    out = np.zeros(h.shape[0], np.uint16)
    lib().orc_rmsnorm_bf16(_p(h, _f64p), h.shape[0], float(eps), _p(out, _u16p))
    return out


def lm_head(W: NVFP4, x_bf16):
    """W one matrix [1, V, H]; x bf16 [B, H] -> (logits fp64 [B, V], argmax [B])."""
    x = _bits16(x_bf16)
    if x.ndim == 1:
        x = x[None]
    B, H = x.shape
    _, V, Hw = W.shape
    assert Hw == H
    logits = np.zeros((B, V), np.float64)
    am = np.zeros(B, np.int32)
    cw = W.c()
    lib().orc_lm_head(ctypes.byref(cw), V, H, _p(x, _u16p), B, _p(logits, _f64p),
                      _p(am, _i32p))
    return logits, am


def sample(logits_f32, temperature: float, top_k: int, top_p: float, u: float):
    """(vocabulary index, kept prefix size m) drawn from one row of fp32 logits."""
    lg = np.ascontiguousarray(logits_f32, dtype=np.float32).reshape(-1)
    m = ctypes.c_int(0)
    idx = lib().orc_sample(_p(lg, _f32p), lg.size, float(temperature), int(top_k), float(top_p),
                           float(u), ctypes.byref(m))
    return int(idx), int(m.value)


def expert_order(idx: np.ndarray, n_experts: int):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.zeros(n_experts, np.int32)
    offsets = np.zeros(n_experts, np.int32)
    perm = np.zeros(T * k, np.int32)
    lib().orc_expert_order(_p(idx, _i32p), T, k, n_experts, _p(counts, _i32p),
                           _p(offsets, _i32p), _p(perm, _i32p))
    return counts, offsets, perm
