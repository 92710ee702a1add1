"""Thin Python binding of libflint.so (include/flint.h), same names as the C ABI.

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (PyTorch provides device memory and
streams); the binding passes their device pointers, the current stream and a
workspace.  If the library is missing or cannot be loaded this module raises on
first use -- there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libflint.so")

FLINT_OK = 0
STATUS_NAMES = {0: "FLINT_OK", 1: "FLINT_ERR_INVALID_ARG", 2: "FLINT_ERR_ALIGNMENT",
                3: "FLINT_ERR_SHAPE", 4: "FLINT_ERR_WORKSPACE", 5: "FLINT_ERR_NONFINITE",
                6: "FLINT_ERR_TIMEOUT", 7: "FLINT_ERR_CUDA", 8: "FLINT_ERR_UNSUPPORTED"}
OP_QUANTIZE, OP_MOE_DECODE, OP_MOE_PREFILL, OP_LM_HEAD = 0, 1, 2, 3
MAX_DECODE_TOKENS = 8


class FlintError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (%d)" % (where, STATUS_NAMES.get(status, "?"), status))


class _NVFP4C(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p), ("n_mat", ctypes.c_int),
                ("rows", ctypes.c_int), ("cols", ctypes.c_int)]


class _LayerC(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("expert_width", ctypes.c_int), ("shared_width", ctypes.c_int),
                ("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("gate", _NVFP4C), ("up", _NVFP4C), ("down", _NVFP4C),
                ("sh_gate", _NVFP4C), ("sh_up", _NVFP4C), ("sh_down", _NVFP4C),
                ("mma_scales", ctypes.c_void_p * 6), ("router_score", ctypes.c_int)]

ROUTER_SOFTMAX, ROUTER_SIGMOID = 0, 1


_lib = None

_SYMBOLS = ["flint_quantize_nvfp4", "flint_dequantize_nvfp4", "flint_nvfp4_mma_scales",
            "flint_sample_logits", "flint_moe_decode", "flint_decode_tokens",
            "flint_decode_tokens_trace", "flint_decode_tokens_noalloc", "flint_moe_prefill",
            "flint_lm_head", "flint_workspace_bytes", "flint_last_device_status",
            "flint_status_string", "flint_version", "flint_set_wait_limit_ns",
            "flint_debug_hold_next_launch", "flint_bench_fp4_mma", "flint_decode_tokens_sample"]


def lib() -> ctypes.CDLL:
    """Load libflint.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libflint.so not built (%s); run python -m "
                          "sparse_moe_decode_02_b300.build" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.flint_quantize_nvfp4.argtypes = [vp, i, i, i, vp, vp, vp, vp, sz, vp]
    L.flint_dequantize_nvfp4.argtypes = [ctypes.POINTER(_NVFP4C), vp, vp]
    L.flint_nvfp4_mma_scales.argtypes = [ctypes.POINTER(_NVFP4C), vp, vp]
    L.flint_decode_tokens.argtypes = [ctypes.POINTER(_LayerC), i, ctypes.POINTER(_NVFP4C), vp, vp,
                                      i, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flint_decode_tokens_trace.argtypes = [ctypes.POINTER(_LayerC), i, ctypes.POINTER(_NVFP4C),
                                            vp, vp, i, ctypes.c_float, vp, vp, vp, vp, vp, vp,
                                            vp, vp, vp, sz, vp]
    L.flint_decode_tokens_sample.argtypes = [ctypes.POINTER(_LayerC), i, ctypes.POINTER(_NVFP4C),
                                             vp, vp, i, ctypes.c_float, ctypes.c_float, i,
                                             ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                             sz, vp]
    L.flint_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.flint_debug_hold_next_launch.argtypes = [i]
    L.flint_decode_tokens_noalloc.argtypes = [ctypes.POINTER(_LayerC), i, ctypes.POINTER(_NVFP4C),
                                              vp, vp, i, ctypes.c_float, vp, vp, vp, vp, vp, vp,
                                              vp]
    L.flint_moe_decode.argtypes = [ctypes.POINTER(_LayerC), vp, vp, vp, vp, ctypes.c_float, vp,
                                   vp, i, vp, sz, vp]
    L.flint_moe_prefill.argtypes = [ctypes.POINTER(_LayerC), vp, vp, vp, vp, vp, vp, i, vp, sz,
                                    vp]
    L.flint_lm_head.argtypes = [ctypes.POINTER(_NVFP4C), vp, vp, vp, i, vp, sz, vp]
    L.flint_sample_logits.argtypes = [vp, i, i, ctypes.c_float, i, ctypes.c_float, vp, vp, vp]
    L.flint_bench_fp4_mma.argtypes = [i, i, i, vp, vp]
    L.flint_workspace_bytes.argtypes = [i] * 8
    L.flint_workspace_bytes.restype = sz
    L.flint_last_device_status.argtypes = [vp]
    L.flint_status_string.argtypes = [i]
    L.flint_status_string.restype = ctypes.c_char_p
    L.flint_version.restype = ctypes.c_char_p
    for name in ("flint_quantize_nvfp4", "flint_dequantize_nvfp4", "flint_nvfp4_mma_scales",
                 "flint_moe_decode", "flint_decode_tokens", "flint_decode_tokens_trace",
                 "flint_decode_tokens_noalloc", "flint_moe_prefill", "flint_lm_head",
                 "flint_last_device_status", "flint_sample_logits", "flint_set_wait_limit_ns",
                 "flint_debug_hold_next_launch", "flint_bench_fp4_mma",
                 "flint_decode_tokens_sample"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != FLINT_OK:
        raise FlintError(status, where)


def workspace_bytes(op, hidden=0, n_experts=0, top_k=0, width=0, shared_width=0, vocab=0,
                    n_tokens=0) -> int:
    return int(lib().flint_workspace_bytes(op, hidden, n_experts, top_k, width, shared_width,
                                           vocab, n_tokens))


def _workspace(nbytes: int, device, ws=None):
    if ws is not None:
        assert ws.numel() >= nbytes and ws.data_ptr() % 256 == 0
        return ws
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


@dataclass
class NVFP4:
    """An NVFP4 stack on the device: codes [n, R, C/2] u8, scales [n, R, C/16] u8, tsc [n]."""
    codes: torch.Tensor
    scales: torch.Tensor
    tsc: torch.Tensor

    @property
    def shape(self):
        n, r, half = self.codes.shape
        return n, r, 2 * half

    def c(self) -> _NVFP4C:
        n, r, c = self.shape
        return _NVFP4C(self.codes.data_ptr(), self.scales.data_ptr(), self.tsc.data_ptr(), n, r, c)

    def nbytes(self) -> int:
        return self.codes.numel() + self.scales.numel() + 4 * self.tsc.numel()


@dataclass
class MoELayer:
    router_w: torch.Tensor          # bf16 [E, H]
    router_bias: torch.Tensor | None  # fp32 [E]
    gate: NVFP4
    up: NVFP4
    down: NVFP4
    sh_gate: NVFP4
    sh_up: NVFP4
    sh_down: NVFP4
    top_k: int
    mma_scales: tuple | None = None   # MMA scale copies of gate, up, down, sh_gate, sh_up, sh_down
    router_score: int = 0             # ROUTER_SOFTMAX or ROUTER_SIGMOID

    @property
    def dims(self):
        E, H = self.router_w.shape
        return H, E, self.top_k, self.gate.shape[1], self.sh_gate.shape[1]

    def c(self) -> _LayerC:
        H, E, k, F, Fs = self.dims
        sf = (ctypes.c_void_p * 6)(*([None] * 6 if self.mma_scales is None else
                                     [m.data_ptr() for m in self.mma_scales]))
        return _LayerC(H, E, k, F, Fs, self.router_w.data_ptr(),
                       None if self.router_bias is None else self.router_bias.data_ptr(),
                       self.gate.c(), self.up.c(), self.down.c(), self.sh_gate.c(),
                       self.sh_up.c(), self.sh_down.c(), sf, self.router_score)

    def nbytes(self) -> int:
        return (self.router_w.numel() * 2 + sum(m.nbytes() for m in (
            self.gate, self.up, self.down, self.sh_gate, self.sh_up, self.sh_down)))


# ------------------------------------------------------------------------- entry points
def quantize_nvfp4(w: torch.Tensor, stream=None, ws=None) -> NVFP4:
    """bf16 [n, R, C] (or [R, C]) CUDA tensor -> NVFP4 stack."""
    if w.dim() == 2:
        w = w.unsqueeze(0)
    assert w.dtype == torch.bfloat16 and w.is_cuda and w.is_contiguous()
    n, r, c = w.shape
    dev = w.device
    q = NVFP4(torch.empty(n, r, c // 2, dtype=torch.uint8, device=dev),
              torch.empty(n, r, c // 16, dtype=torch.uint8, device=dev),
              torch.empty(n, dtype=torch.float32, device=dev))
    nb = workspace_bytes(OP_QUANTIZE, n_tokens=n)
    ws = _workspace(nb, dev, ws)
    _check(lib().flint_quantize_nvfp4(_ptr(w), n, r, c, _ptr(q.codes), _ptr(q.scales),
                                      _ptr(q.tsc), _ptr(ws), ws.numel(), _stream(stream)),
           "flint_quantize_nvfp4")
    return q


def nvfp4_mma_scales(m: NVFP4, stream=None) -> torch.Tensor:
    """MMA scale copy of an NVFP4 stack's block scales (see flint.h)."""
    out = torch.empty_like(m.scales)
    mc = m.c()
    _check(lib().flint_nvfp4_mma_scales(ctypes.byref(mc), _ptr(out), _stream(stream)),
           "flint_nvfp4_mma_scales")
    return out


def bench_fp4_mma(mode: int, iters: int, ctas: int, stream=None) -> torch.Tensor:
    """Launch the block-scaled FP4 MMA microbenchmark (see flint.h); returns the
    per-CTA cycle counts (device int64 tensor, filled when the stream reaches it)."""
    cyc = torch.zeros(ctas, dtype=torch.int64, device="cuda")
    _check(lib().flint_bench_fp4_mma(mode, iters, ctas, _ptr(cyc), _stream(stream)),
           "flint_bench_fp4_mma")
    return cyc


def dequantize_nvfp4(m: NVFP4, stream=None) -> torch.Tensor:
    n, r, c = m.shape
    out = torch.empty(n, r, c, dtype=torch.float32, device=m.codes.device)
    mc = m.c()
    _check(lib().flint_dequantize_nvfp4(ctypes.byref(mc), _ptr(out), _stream(stream)),
           "flint_dequantize_nvfp4")
    return out


def moe_decode(layer: MoELayer, x: torch.Tensor, residual: torch.Tensor | None = None,
               out: torch.Tensor | None = None, x_next: torch.Tensor | None = None,
               rms_eps: float = 1e-6, topk_idx: torch.Tensor | None = None,
               topk_w: torch.Tensor | None = None, ws: torch.Tensor | None = None,
               stream=None):
    """One MoE layer for B tokens; returns out (fp32 [B, H])."""
    if x.dim() == 1:
        x = x.unsqueeze(0)
    B = x.shape[0]
    H, E, k, F, Fs = layer.dims
    if out is None:
        out = torch.empty(B, H, dtype=torch.float32, device=x.device)
    nb = workspace_bytes(OP_MOE_DECODE, H, E, k, F, Fs, 0, B)
    ws = _workspace(nb, x.device, ws)
    lc = layer.c()
    _check(lib().flint_moe_decode(ctypes.byref(lc), _ptr(x), _ptr(residual), _ptr(out),
                                  _ptr(x_next), float(rms_eps), _ptr(topk_idx), _ptr(topk_w), B,
                                  _ptr(ws), ws.numel(), _stream(stream)), "flint_moe_decode")
    return out


def decode_tokens(layers, x: torch.Tensor, head: NVFP4 | None = None,
                  residual: torch.Tensor | None = None, rms_eps: float = 1e-6, out=None,
                  x_out=None, logits=None, argmax=None, topk_idx=None, topk_w=None, ws=None,
                  stream=None, x_trace=None, h_trace=None):
    """T tokens through len(layers) chained layers (+ head) in one launch.  With x_trace
    (bf16 [T, L, H]) or h_trace (fp32 [T, L, H]) the call is flint_decode_tokens_trace."""
    if x.dim() == 1:
        x = x.unsqueeze(0)
    T = x.shape[0]
    H, E, k, F, Fs = layers[0].dims
    arr = (_LayerC * len(layers))(*[l.c() for l in layers])
    hc = head.c() if head is not None else None
    nb = workspace_bytes(OP_MOE_DECODE, H, E, k, F, Fs, 0, T)
    ws = _workspace(nb, x.device, ws)
    common = (arr, len(layers), ctypes.byref(hc) if hc else None, _ptr(x), _ptr(residual), T,
              float(rms_eps), _ptr(out), _ptr(x_out), _ptr(logits), _ptr(argmax),
              _ptr(topk_idx), _ptr(topk_w))
    if x_trace is None and h_trace is None:
        _check(lib().flint_decode_tokens(*common, _ptr(ws), ws.numel(), _stream(stream)),
               "flint_decode_tokens")
    else:
        _check(lib().flint_decode_tokens_trace(*common, _ptr(x_trace), _ptr(h_trace), _ptr(ws),
                                               ws.numel(), _stream(stream)),
               "flint_decode_tokens_trace")


def decode_tokens_sample(layers, x: torch.Tensor, head: NVFP4, uniforms: torch.Tensor,
                         temperature: float = 1.0, top_k: int = 20, top_p: float = 0.95,
                         tokens=None, residual=None, rms_eps: float = 1e-6, out=None, x_out=None,
                         logits=None, argmax=None, topk_idx=None, topk_w=None, ws=None,
                         stream=None) -> torch.Tensor:
    """decode_tokens with each token drawn from the head's logits inside the launch
    (flint_decode_tokens_sample); returns tokens (int32 [T])."""
    if x.dim() == 1:
        x = x.unsqueeze(0)
    T = x.shape[0]
    H, E, k, F, Fs = layers[0].dims
    if tokens is None:
        tokens = torch.empty(T, dtype=torch.int32, device=x.device)
    arr = (_LayerC * len(layers))(*[l.c() for l in layers])
    hc = head.c()
    nb = workspace_bytes(OP_MOE_DECODE, H, E, k, F, Fs, 0, T)
    ws = _workspace(nb, x.device, ws)
    _check(lib().flint_decode_tokens_sample(arr, len(layers), ctypes.byref(hc), _ptr(x),
                                            _ptr(residual), T, float(rms_eps), float(temperature),
                                            int(top_k), float(top_p), _ptr(uniforms), _ptr(tokens),
                                            _ptr(out), _ptr(x_out), _ptr(logits), _ptr(argmax),
                                            _ptr(topk_idx), _ptr(topk_w), _ptr(ws), ws.numel(),
                                            _stream(stream)), "flint_decode_tokens_sample")
    return tokens


def set_wait_limit_ns(ns: int) -> None:
    """Bound of every device-side wait (0 restores the 2 s default)."""
    _check(lib().flint_set_wait_limit_ns(int(ns)), "flint_set_wait_limit_ns")


def debug_hold_next_launch(what: int) -> None:
    """Arms the next decode (1) or prompt (2) launch of this thread to withhold one
    hand-over, so that its waits run out (a fault-handling test aid; 0 disarms)."""
    _check(lib().flint_debug_hold_next_launch(int(what)), "flint_debug_hold_next_launch")


def decode_tokens_noalloc(layers, x: torch.Tensor, head: NVFP4 | None = None,
                          residual: torch.Tensor | None = None, rms_eps: float = 1e-6, out=None,
                          x_out=None, logits=None, argmax=None, topk_idx=None, topk_w=None,
                          stream=None):
    """decode_tokens with the library's fixed device scratch instead of a workspace (for
    callers that cannot allocate; see flint_decode_tokens_noalloc in flint.h)."""
    if x.dim() == 1:
        x = x.unsqueeze(0)
    arr = (_LayerC * len(layers))(*[l.c() for l in layers])
    hc = head.c() if head is not None else None
    _check(lib().flint_decode_tokens_noalloc(arr, len(layers), ctypes.byref(hc) if hc else None,
                                             _ptr(x), _ptr(residual), x.shape[0], float(rms_eps),
                                             _ptr(out), _ptr(x_out), _ptr(logits), _ptr(argmax),
                                             _ptr(topk_idx), _ptr(topk_w), _stream(stream)),
           "flint_decode_tokens_noalloc")


def moe_prefill(layer: MoELayer, x: torch.Tensor, out: torch.Tensor | None = None,
                topk_idx=None, topk_w=None, expert_counts=None, pair_order=None, ws=None,
                stream=None):
    T = x.shape[0]
    H, E, k, F, Fs = layer.dims
    if out is None:
        out = torch.empty(T, H, dtype=torch.float32, device=x.device)
    nb = workspace_bytes(OP_MOE_PREFILL, H, E, k, F, Fs, 0, T)
    ws = _workspace(nb, x.device, ws)
    lc = layer.c()
    _check(lib().flint_moe_prefill(ctypes.byref(lc), _ptr(x), _ptr(out), _ptr(topk_idx),
                                   _ptr(topk_w), _ptr(expert_counts), _ptr(pair_order), T,
                                   _ptr(ws), ws.numel(), _stream(stream)), "flint_moe_prefill")
    return out


def lm_head(W: NVFP4, x: torch.Tensor, logits: torch.Tensor | None = None,
            argmax: torch.Tensor | None = None, want_logits: bool = True, ws=None, stream=None):
    """Returns (logits fp32 [B, V] or None, argmax int32 [B])."""
    if x.dim() == 1:
        x = x.unsqueeze(0)
    B = x.shape[0]
    _, V, H = W.shape
    if logits is None and want_logits:
        logits = torch.empty(B, V, dtype=torch.float32, device=x.device)
    if argmax is None:
        argmax = torch.empty(B, dtype=torch.int32, device=x.device)
    nb = workspace_bytes(OP_LM_HEAD, H, 0, 0, 0, 0, V, B)
    ws = _workspace(nb, x.device, ws)
    wc = W.c()
    _check(lib().flint_lm_head(ctypes.byref(wc), _ptr(x), _ptr(logits), _ptr(argmax), B, _ptr(ws),
                               ws.numel(), _stream(stream)), "flint_lm_head")
    return logits, argmax


def last_device_status(stream=None) -> int:
    return int(lib().flint_last_device_status(_stream(stream)))


def status_string(status: int) -> str:
    return lib().flint_status_string(int(status)).decode()


def version() -> str:
    return lib().flint_version().decode()


def sample_logits(logits: torch.Tensor, uniforms: torch.Tensor, temperature: float = 1.0,
                  top_k: int = 20, top_p: float = 0.95, stream=None) -> torch.Tensor:
    """One token per row of fp32 logits [B, V] (top-k, temperature, top-p; see flint.h),
    drawn with the caller's uniforms fp32 [B] in [0, 1).  Returns int32 [B]."""
    assert logits.dtype == torch.float32 and logits.is_cuda and logits.is_contiguous()
    B, V = logits.shape
    u = uniforms.to(device=logits.device, dtype=torch.float32).contiguous()
    out = torch.empty(B, dtype=torch.int32, device=logits.device)
    _check(lib().flint_sample_logits(_ptr(logits), B, V, float(temperature), int(top_k),
                                     float(top_p), _ptr(u), _ptr(out), _stream(stream)),
           "flint_sample_logits")
    return out
