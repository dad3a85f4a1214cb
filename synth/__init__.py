"""Seeded synthetic inputs for the MoE layer forward.

This module is shared by both sides of every parity test: the CPU oracle
(``oracle/``) and the CUDA library's tests and benchmark.  It draws token
embeddings, router weights, expert weights and the per-expert router offsets
that the workloads call for, and it holds no step of the MoE computation
itself (no routing, no top-k, no softmax, no FFN, no combine).

Generator.  Value ``i`` of a tensor is a pure function of
``(seed, layer, tensor_id, i)``: a counter-based generator.  Two 32-bit words
are drawn per value from a keyed double application of the MurmurHash3 32-bit
finaliser ("fmix32", Appleby, MurmurHash3 reference code), mapped to uniforms
``u = (r + 0.5) / 2**32`` in (0, 1), and turned into one standard normal by
the Box-Muller transform ``sqrt(-2 ln u1) * cos(2 pi u2)`` (Box & Muller,
1958).  All integer steps are exact on any device, so a slice of a tensor can
be regenerated on the CPU or on the GPU without drawing the rest; the float64
``log``/``cos``/``sqrt`` may differ by an ulp between devices, which changes
the float32 (or bfloat16) result with probability about 2**-29 (2**-44) per
value.  Parity tests that need full-size tensors on both sides generate them
once and copy them, so they never depend on that.

Workloads (shapes and value distributions of the five layer configurations):

* ``x ~ N(0, 1)``; every weight ``~ N(0, std = 1/sqrt(fan_in))`` with
  ``fan_in = d_model`` for the router, gate and up projections and
  ``fan_in = d_ff`` for the down projection.
* Qwen2-MoE-shaped layer: router logits offset per expert by
  ``-1.1 * ln(e + 1)``, the log of a Zipf(s=1.1) pmf up to a constant, so
  expert 0 is the hottest.
* DeepSeek-MoE-shaped layer, masked run: experts ``e % 4 == 3`` get an
  offset of ``-inf`` (25 % of the experts receive no token).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

_MASK32 = 0xFFFFFFFF
_CHUNK = 1 << 24

# tensor ids inside one layer
X, W_ROUTER, W_GATE, W_UP, W_DOWN = 0, 1, 2, 3, 4


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for int64 x in [0, 2**32) without int64 overflow."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _MASK32


def _fmix32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x85EBCA6B)
    x = x ^ (x >> 13)
    x = _mul32(x, 0xC2B2AE35)
    x = x ^ (x >> 16)
    return x


def _fmix32_int(x: int) -> int:
    x &= _MASK32
    x ^= x >> 16
    x = (x * 0x85EBCA6B) & _MASK32
    x ^= x >> 13
    x = (x * 0xC2B2AE35) & _MASK32
    x ^= x >> 16
    return x


def _keys(seed: int, layer: int, tensor_id: int) -> tuple[int, int, int, int]:
    base = _fmix32_int(seed * 0x9E3779B1 + 0x7F4A7C15)
    base = _fmix32_int(base ^ (layer * 0x85EBCA77 + 0x165667B1))
    base = _fmix32_int(base ^ (tensor_id * 0xC2B2AE3D + 0x27D4EB2F))
    ks = []
    for j in range(4):
        base = _fmix32_int(base + 0x9E3779B9)
        ks.append(base)
    return ks[0], ks[1], ks[2], ks[3]


def normal_f64(start: int, count: int, seed: int, layer: int, tensor_id: int,
               device="cpu") -> torch.Tensor:
    """Standard normals for indices [start, start+count) of one tensor, float64."""
    if start < 0 or start + count > (1 << 32):
        raise ValueError("tensor index out of the generator's 2**32 range")
    k1, k2, k3, k4 = _keys(seed, layer, tensor_id)
    i = torch.arange(start, start + count, dtype=torch.int64, device=device)
    r1 = _fmix32((_fmix32((i + k1) & _MASK32) + k2) & _MASK32)
    r2 = _fmix32((_fmix32((i + k3) & _MASK32) + k4) & _MASK32)
    del i
    scale = 1.0 / 4294967296.0
    u1 = (r1.to(torch.float64) + 0.5) * scale
    u2 = (r2.to(torch.float64) + 0.5) * scale
    del r1, r2
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def normal(shape, seed: int, layer: int, tensor_id: int, std: float = 1.0,
           dtype=torch.float32, device="cpu") -> torch.Tensor:
    """A tensor of N(0, std^2) values, rounded (RNE) to ``dtype``.

    float64 -> float32 -> (bfloat16) rounding, each step round-to-nearest-even.
    """
    shape = tuple(int(s) for s in shape)
    n = 1
    for s in shape:
        n *= s
    out = torch.empty(n, dtype=dtype, device=device)
    for s0 in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s0)
        v = normal_f64(s0, c, seed, layer, tensor_id, device) * std
        out[s0:s0 + c] = v.to(torch.float32).to(dtype)
    return out.view(shape)


@dataclass(frozen=True)
class LayerShape:
    """Shape and recipe of one MoE layer workload."""
    name: str
    d_model: int
    d_ff: int
    n_experts: int
    top_k: int
    dtype: str                 # "fp32" or "bf16"
    bias: str = "none"         # "none" | "zipf" | "mask4"
    zipf_s: float = 1.1

    def with_bias(self, bias: str) -> "LayerShape":
        return replace(self, bias=bias)


TINY = LayerShape("tiny", 128, 256, 8, 2, "fp32")
MIXTRAL = LayerShape("mixtral", 4096, 14336, 8, 2, "bf16")
QWEN2 = LayerShape("qwen2_moe", 2048, 1408, 64, 2, "bf16", bias="zipf")
DEEPSEEK = LayerShape("deepseek_moe", 2048, 1408, 128, 4, "bf16")
DEEPSEEK_MASKED = DEEPSEEK.with_bias("mask4")

SHAPES = {s.name: s for s in (TINY, MIXTRAL, QWEN2, DEEPSEEK)}

# token counts each workload is run at
TOKENS = {
    "tiny": (16,),
    "mixtral": (1, 16, 128, 4096),
    "qwen2_moe": (1, 64, 2048, 8192),
    "deepseek_moe": (16384,),
}

STACK_LAYERS = 32
STACK_BATCHES = (1, 8, 64)
STACK_EPS = 1e-5


def torch_dtype(shape: LayerShape):
    return torch.float32 if shape.dtype == "fp32" else torch.bfloat16


def router_offset(shape: LayerShape) -> Optional[torch.Tensor]:
    """Per-expert logit offset [E] float32 (None when the workload has none)."""
    E = shape.n_experts
    if shape.bias == "none":
        return None
    e = torch.arange(E, dtype=torch.float64)
    if shape.bias == "zipf":
        return (-shape.zipf_s * torch.log(e + 1.0)).to(torch.float32)
    if shape.bias == "mask4":
        b = torch.zeros(E, dtype=torch.float32)
        b[(torch.arange(E) % 4) == 3] = float("-inf")
        return b
    raise ValueError(f"unknown offset recipe {shape.bias!r}")


def tokens(shape: LayerShape, T: int, seed: int, layer: int = 0,
           device="cpu") -> torch.Tensor:
    """Token embeddings x [T, d_model], N(0,1)."""
    return normal((T, shape.d_model), seed, layer, X, 1.0, torch_dtype(shape), device)


def router_weight(shape: LayerShape, seed: int, layer: int = 0, device="cpu"):
    """W_r [d_model, E], N(0, 1/d_model)."""
    return normal((shape.d_model, shape.n_experts), seed, layer, W_ROUTER,
                  1.0 / math.sqrt(shape.d_model), torch_dtype(shape), device)


def expert_weights(shape: LayerShape, seed: int, layer: int = 0, device="cpu"):
    """(W_gate [E,d,f], W_up [E,d,f], W_down [E,f,d]) in the library's input layout."""
    E, d, f = shape.n_experts, shape.d_model, shape.d_ff
    dt = torch_dtype(shape)
    wg = normal((E, d, f), seed, layer, W_GATE, 1.0 / math.sqrt(d), dt, device)
    wu = normal((E, d, f), seed, layer, W_UP, 1.0 / math.sqrt(d), dt, device)
    wd = normal((E, f, d), seed, layer, W_DOWN, 1.0 / math.sqrt(f), dt, device)
    return wg, wu, wd


def layer(shape: LayerShape, T: int, seed: int, layer_idx: int = 0, device="cpu"):
    """All inputs of one layer call as a dict of tensors (library input layout)."""
    wg, wu, wd = expert_weights(shape, seed, layer_idx, device)
    return {
        "x": tokens(shape, T, seed, layer_idx, device),
        "w_router": router_weight(shape, seed, layer_idx, device),
        "router_bias": router_offset(shape),
        "w_gate": wg, "w_up": wu, "w_down": wd,
    }
