"""Seeded synthetic inputs for the Flint MoE feed-forward / output-head path.

This module is the one piece both sides share: the tests feed the same tensors to
the CUDA library and to the CPU oracle, and the benchmark uses it to build its
workloads.  It holds none of the method's arithmetic (no quantisation, routing or
products) and imports neither the library binding nor the oracle.

Generator.  Every value is a pure function of (seed, tensor id, element index), so
any slice of any tensor can be regenerated on either device and comes out bit for
bit the same:

    h = mix(mix(i ^ k0) ^ k1)                  32-bit counter hash ("lowbias32" by
                                               C. Wellons), i = element index,
                                               (k0, k1) = 64-bit SplitMix64 key
    v = NORMAL_TABLE[h >> 16] * sigma          65,536-entry inverse-normal table:
                                               Phi^-1((u + 1/2) / 65536), rounded
                                               to bf16 after the sigma multiply

All integer steps stay inside int64 without overflow, so CPU and CUDA tensors
agree exactly.  The table is built once on the host in fp64 (scipy's ndtri).

The distributions follow the workload description of the Flint pages ("Flint: 125
tokens a second is what 2.5B active parameters buy at 273 GB/s", section "The
shape, read from the headers"): weights N(0, 0.02), activations N(0, 1), and, for
skewed routing, a per-expert router bias -s*ln(rank) from a seeded permutation of
ranks 1..E (the log of a Zipf(s) popularity, up to a constant).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_MASK32 = 0xFFFFFFFF
_MASK64 = 0xFFFFFFFFFFFFFFFF


def splitmix64(x: int) -> int:
    """One SplitMix64 step (S. Vigna), on Python ints."""
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def tensor_key(seed: int, *ids: int) -> int:
    """64-bit key of a tensor: SplitMix64 folded over (seed, ids...)."""
    k = splitmix64(seed & _MASK64)
    for i in ids:
        k = splitmix64(k ^ (int(i) & _MASK64))
    return k


# tensor kinds (part of the key)
KIND_ROUTER, KIND_GATE, KIND_UP, KIND_DOWN = 1, 2, 3, 4
KIND_SH_GATE, KIND_SH_UP, KIND_SH_DOWN = 5, 6, 7
KIND_X, KIND_HEAD, KIND_BIAS = 8, 9, 10


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for 0 <= x < 2^32, without leaving int64."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + ((x * hi) & 0xFFFF) * 65536) & _MASK32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    return x ^ (x >> 16)


_TABLES: dict = {}


def _normal_table_bf16(sigma: float, device) -> torch.Tensor:
    """bf16(sigma * Phi^-1((u + 0.5)/65536)) for u in [0, 65536), built on the host
    (so every device holds the same bits), then moved to `device`."""
    key = (float(sigma), str(device))
    if key not in _TABLES:
        from scipy.special import ndtri
        u = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
        host = torch.from_numpy(ndtri(u) * float(sigma)).to(torch.bfloat16)
        _TABLES[key] = host.to(device)
    return _TABLES[key]


def hash_u32(key: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """32-bit counter hashes for element indices [start, start + n) (int64 tensor)."""
    k0, k1 = key & _MASK32, (key >> 32) & _MASK32
    i = torch.arange(start, start + n, dtype=torch.int64, device=device) & _MASK32
    return _mix32(_mix32(i ^ k0) ^ k1)


def normal_bf16(key: int, n: int, sigma: float, start: int = 0, device="cpu",
                chunk: int = 1 << 25) -> torch.Tensor:
    """n bf16 draws of N(0, sigma^2) for element indices [start, start + n)."""
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    table = _normal_table_bf16(sigma, device)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        h = hash_u32(key, start + s, m, device)
        out[s:s + m] = table[h >> 16]
    return out


def zipf_bias(seed: int, n_experts: int, s: float = 1.1, layer: int = 0) -> np.ndarray:
    """fp32 [E] router bias -s*ln(rank): a seeded permutation of ranks 1..E."""
    key = tensor_key(seed, layer, KIND_BIAS)
    h = hash_u32(key, 0, n_experts).numpy()
    ranks = np.empty(n_experts, np.int64)
    ranks[np.argsort(h, kind="stable")] = np.arange(1, n_experts + 1)
    return (-s * np.log(ranks.astype(np.float64))).astype(np.float32)


# --------------------------------------------------------------------------- workloads
@dataclass(frozen=True)
class MoeShape:
    hidden: int
    n_experts: int
    top_k: int
    expert_width: int
    shared_width: int
    vocab: int = 0


TINY = MoeShape(hidden=256, n_experts=16, top_k=2, expert_width=64, shared_width=128,
                vocab=4096)
FLINT = MoeShape(hidden=2048, n_experts=256, top_k=6, expert_width=512, shared_width=1024,
                 vocab=150144)

# One of the model's dense SwiGLU layers ("Flint: 125 tokens a second is what 2.5B active
# parameters buy at 273 GB/s", section "Built from scratch?": width 6,144): no router,
# no routed experts; the block is the layer's shared matrices.
FLINT_DENSE = MoeShape(hidden=2048, n_experts=0, top_k=0, expert_width=0, shared_width=6144,
                       vocab=150144)

W_SIGMA = 0.02
X_SIGMA = 1.0


@dataclass
class LayerSpec:
    """Which tensors make one layer: keys and shapes, no values."""
    shape: MoeShape
    seed: int
    layer: int = 0
    zipf: float | None = None          # router bias exponent, None = no bias
    router_score: int = 0              # 0 softmax, 1 sigmoid scoring (a layer flag)

    def key(self, kind: int) -> int:
        return tensor_key(self.seed, self.layer, kind)

    def dims(self, kind: int):
        s = self.shape
        return {KIND_ROUTER: (1, s.n_experts, s.hidden),
                KIND_GATE: (s.n_experts, s.expert_width, s.hidden),
                KIND_UP: (s.n_experts, s.expert_width, s.hidden),
                KIND_DOWN: (s.n_experts, s.hidden, s.expert_width),
                KIND_SH_GATE: (1, s.shared_width, s.hidden),
                KIND_SH_UP: (1, s.shared_width, s.hidden),
                KIND_SH_DOWN: (1, s.hidden, s.shared_width)}[kind]

    def weights_bf16(self, kind: int, device="cpu", experts=None) -> torch.Tensor:
        """bf16 [n, R, C] of one stack; `experts` picks a subset of matrices."""
        n, r, c = self.dims(kind)
        per = r * c
        key = self.key(kind)
        if experts is None:
            return normal_bf16(key, n * per, W_SIGMA, 0, device).view(n, r, c)
        parts = [normal_bf16(key, per, W_SIGMA, int(e) * per, device) for e in experts]
        return torch.stack(parts).view(len(parts), r, c)

    def bias(self):
        if self.zipf is None:
            return None
        return zipf_bias(self.seed, self.shape.n_experts, self.zipf, self.layer)


def tokens_bf16(seed: int, hidden: int, n_tok: int, start_tok: int = 0, stream: int = 0,
                device="cpu") -> torch.Tensor:
    """bf16 [n_tok, hidden] N(0,1) activations; token t is the same in any slice."""
    key = tensor_key(seed, stream, KIND_X)
    return normal_bf16(key, n_tok * hidden, X_SIGMA, start_tok * hidden, device).view(
        n_tok, hidden)


def head_bf16(seed: int, vocab: int, hidden: int, device="cpu", rows=None) -> torch.Tensor:
    """bf16 [1, V, H] output-head weights, or rows [r0, r1) of them."""
    key = tensor_key(seed, 0, KIND_HEAD)
    if rows is None:
        return normal_bf16(key, vocab * hidden, W_SIGMA, 0, device).view(1, vocab, hidden)
    r0, r1 = rows
    return normal_bf16(key, (r1 - r0) * hidden, W_SIGMA, r0 * hidden, device).view(
        1, r1 - r0, hidden)
