"""Seeded synthetic inputs for the routed-MoE layer.

This module only draws numbers: it holds none of the layer's arithmetic and
imports neither the CUDA binding nor the CPU oracle, so both sides can be fed
the very same bytes (generate once, copy to wherever each side runs).

Distributions (the Qwen3-30B-A3B / Qwen3-235B-A22B shapes with seeded random
weights; no checkpoint is used):
  * hidden state x ~ N(0, 1), rounded to bf16;
  * router weight ~ N(0, 0.02), bf16, [E, D];
  * SMOE-Q4 codes uniform in 0..15 (so every byte, two codes, is uniform in
    0..255), scale = bf16(|N(0, 0.02)| / 8), bias = -8 * scale (exact in bf16),
    one scale and one bias per group of 64 along the input dimension;
  * RMSNorm gain of ones when a norm is requested;
  * SMOE-Q2 (code_bits=2): codes uniform in 0..3 (every byte, four codes,
    uniform in 0..255), scale = bf16(|N(0, 0.02)| / 2), bias = -2 * scale
    (exact), so a weight has about the spread of the Q4 draw.

Storage layout (fixed by this project): codes row-major [rows, cols/2] with
element 2j in the low nibble of byte j and 2j+1 in the high nibble; scales and
biases [rows, cols/64]; gate and up [E, F, D]; down [E, D, F].  SMOE-Q2 codes
are [rows, cols/4], element 4j+k in bits 2k..2k+1 of byte j.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch

GROUP = 64


@dataclass
class LayerWeights:
    d_model: int
    n_experts: int
    top_k: int
    ffn_dim: int
    router_w: torch.Tensor          # bf16 [E, D]
    gate_q: torch.Tensor            # uint8 [E, F, D/2]
    gate_s: torch.Tensor            # bf16 [E, F, D/64]
    gate_b: torch.Tensor
    up_q: torch.Tensor
    up_s: torch.Tensor
    up_b: torch.Tensor
    down_q: torch.Tensor            # uint8 [E, D, F/2]
    down_s: torch.Tensor            # bf16 [E, D, F/64]
    down_b: torch.Tensor
    rms_gain: Optional[torch.Tensor] = None   # bf16 [D] or None
    rms_eps: float = 1e-6
    norm_topk_prob: bool = True
    code_bits: int = 4                         # 4: SMOE-Q4, 2: SMOE-Q2

    def tensors(self) -> List[torch.Tensor]:
        out = [self.router_w, self.gate_q, self.gate_s, self.gate_b, self.up_q, self.up_s,
               self.up_b, self.down_q, self.down_s, self.down_b]
        if self.rms_gain is not None:
            out.append(self.rms_gain)
        return out

    def nbytes_expert(self) -> int:
        """Bytes of one expert's three Q4 matrices (codes + scales + biases)."""
        per = 0
        for n in ("gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b", "down_q", "down_s",
                  "down_b"):
            t = getattr(self, n)
            per += t[0].numel() * t.element_size()
        return per

    def nbytes_router(self) -> int:
        return self.router_w.numel() * self.router_w.element_size()


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def _scales(shape, g, device, code_bits=4):
    div, mid = (8.0, -8.0) if code_bits == 4 else (2.0, -2.0)
    s = (torch.randn(shape, generator=g, device=device, dtype=torch.float32).abs_() * (0.02 / div)
         ).to(torch.bfloat16)
    return s, (s.float() * mid).to(torch.bfloat16)


def layer_weights(d_model: int, n_experts: int, ffn_dim: int, top_k: int = 8, *, seed: int,
                  device="cpu", rms_norm: bool = False, norm_topk_prob: bool = True,
                  code_bits: int = 4) -> LayerWeights:
    """One layer of seeded weights (see the module docstring)."""
    D, E, F = d_model, n_experts, ffn_dim
    assert D % GROUP == 0 and F % GROUP == 0 and code_bits in (2, 4)
    per_byte = 8 // code_bits
    g = _gen(seed, device)
    router = (torch.randn((E, D), generator=g, device=device) * 0.02).to(torch.bfloat16)

    def codes(rows, cols):
        return torch.randint(0, 256, (E, rows, cols // per_byte), generator=g, device=device,
                             dtype=torch.uint8)

    gq = codes(F, D)
    gs, gb = _scales((E, F, D // GROUP), g, device, code_bits)
    uq = codes(F, D)
    us, ub = _scales((E, F, D // GROUP), g, device, code_bits)
    dq = codes(D, F)
    ds, db = _scales((E, D, F // GROUP), g, device, code_bits)
    gain = torch.ones(D, dtype=torch.bfloat16, device=device) if rms_norm else None
    return LayerWeights(D, E, top_k, F, router, gq, gs, gb, uq, us, ub, dq, ds, db, gain,
                        1e-6, norm_topk_prob, code_bits)


def dense_weights(shape, *, seed: int, device="cpu", std: float = 0.02,
                  row_spread: float = 0.0) -> torch.Tensor:
    """bf16 weights ~ N(0, std^2) of any shape (dense projections, LM head, or
    the bf16 expert weights a quantiser takes); with row_spread > 0 each row's
    std is further multiplied by exp(N(0, row_spread^2)) (rows of very
    different magnitude)."""
    g = _gen(seed, device)
    w = torch.randn(shape, generator=g, device=device) * std
    if row_spread > 0:
        w *= torch.exp(torch.randn(tuple(shape[:-1]) + (1,), generator=g, device=device) * row_spread)
    return w.to(torch.bfloat16)


def hidden(T: int, d_model: int, *, seed: int, device="cpu") -> torch.Tensor:
    """T hidden states ~ N(0, 1) as bf16 [T, D]."""
    g = _gen(seed, device)
    return torch.randn((T, d_model), generator=g, device=device).to(torch.bfloat16)


def correlated_hidden(T: int, d_model: int, alpha: float, *, seed: int, device="cpu"
                      ) -> torch.Tensor:
    """x_t = alpha * s + sqrt(1 - alpha^2) * z_t with one seeded shared direction s.

    Tokens that share a direction route to overlapping experts; alpha sets
    how many distinct experts a chunk reaches (alpha = 0: independent)."""
    g = _gen(seed, device)
    s = torch.randn((1, d_model), generator=g, device=device)
    z = torch.randn((T, d_model), generator=g, device=device)
    return (alpha * s + (1.0 - alpha * alpha) ** 0.5 * z).to(torch.bfloat16)


def overlap_stream(T: int, d_model: int, rho: float, *, seed: int, device="cpu"
                   ) -> torch.Tensor:
    """A decode stream x_{s+1} = rho * x_s + sqrt(1 - rho^2) * z (AR(1)), bf16 [T, D].

    rho sets how many experts consecutive tokens share."""
    g = _gen(seed, device)
    z = torch.randn((T, d_model), generator=g, device=device)
    out = torch.empty_like(z)
    out[0] = z[0]
    c = (1.0 - rho * rho) ** 0.5
    for t in range(1, T):
        out[t] = rho * out[t - 1] + c * z[t]
    return out.to(torch.bfloat16)


def zipf_bias_hidden(T: int, router_w: torch.Tensor, s: float, scale: float, *, seed: int
                     ) -> torch.Tensor:
    """Hidden states whose router logits carry a Zipf(s) bias over a seeded
    expert permutation: x_t = z_t + pinv(Wr) b, so that Wr x_t = Wr z_t + b
    (up to the bf16 rounding of x_t).  `scale` sets the bias amplitude."""
    device = router_w.device
    E, D = router_w.shape
    g = _gen(seed, device)
    perm = torch.randperm(E, generator=g, device=device)
    ranks = torch.empty(E, device=device)
    ranks[perm] = torch.arange(1, E + 1, device=device, dtype=torch.float32)
    b = scale * ranks.pow(-s)
    b = b - b.mean()
    pinv = torch.linalg.pinv(router_w.double()).float()       # [D, E]
    z = torch.randn((T, D), generator=g, device=device)
    return (z + (pinv @ b).unsqueeze(0)).to(torch.bfloat16)


@dataclass
class Stack:
    """A stack of layers that share one shape (a decode or prefill model)."""
    layers: List[LayerWeights] = field(default_factory=list)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for L in self.layers for t in L.tensors())


def stack(n_layers: int, d_model: int, n_experts: int, ffn_dim: int, top_k: int = 8, *,
          seed: int, device="cpu", rms_norm: bool = True) -> Stack:
    return Stack([layer_weights(d_model, n_experts, ffn_dim, top_k, seed=seed * 1000 + i,
                                device=device, rms_norm=rms_norm) for i in range(n_layers)])
