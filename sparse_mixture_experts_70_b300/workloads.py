"""Seeded synthetic workloads for the top-k MoE FFN layer forward.

This module only draws random inputs; it holds none of the layer's arithmetic. Both the CUDA path
(through the C-ABI binding) and the double-precision oracle read the tensors it returns, byte for
byte.

Shapes and layouts (row-major throughout):
  h    [T, d]     activations, f32 or bf16
  W_r  [d, E]     router weight, always f32 (the router runs in f32 even when the rest is bf16,
                  "selective precision" in arjunjaggi.com "Mixture of Experts in LLMs", section
                  "Switch Transformers"; the lensaml.com explainer, Step 2, prints it as 4096 x 8)
  b_r  [E]        optional f32 router bias (only the many-small-experts workload has one)
  W1   [E, f, d]  first projection, out x in (K-contiguous)
  W3   [E, f, d]  gate projection of the SwiGLU form (absent for the GELU form)
  W2   [E, d, f]  second projection, out x in
  b1   [E, f], b2 [E, d]  f32 biases (only the micro workload has them; zero-initialised)

Draw order (one torch CPU generator per workload, seeded): h, W_r, b_r, then for each expert e in
order W1[e], W3[e] (SwiGLU only), W2[e]. Every draw is torch.randn in f32, scaled by the standard
deviation in f32, then rounded to bf16 (round to nearest even) where the workload is bf16.
Weights ~ N(0, 1/fan_in); h ~ N(0, 1); the router bias ~ N(0, variance 2).
"""
from __future__ import annotations

import dataclasses
import math

import torch

ACT_GELU_TANH = "gelu_tanh"
ACT_SWIGLU = "swiglu"
GATE_RENORM = "renorm"
GATE_RAW_PROB = "raw_prob"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    act: str
    gate: str
    dtype: str            # "f32" or "bf16": the storage type of h, expert weights, H and y
    has_bias: bool        # expert biases b1, b2 (zero-initialised but applied)
    router_bias_var: float | None
    seed: int
    capacity_factor: float = 0.0  # > 0: each expert keeps at most floor(factor T k / E) slots
    fuse_gather: bool = False     # the layer call reads expert rows of h without a permuted copy
    sel_bias_std: float = 0.0     # > 0: a selection-only routing bias b ~ N(0, std^2) per expert

    @property
    def P(self) -> int:
        """Routing slots: every token is copied to k experts."""
        return self.T * self.k

    @property
    def n_mats(self) -> int:
        return 3 if self.act == ACT_SWIGLU else 2

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def expert_flops(self) -> int:
        """Multiply-add work of the grouped expert FFN, counted as 2 flops per MAC."""
        return 2 * self.P * self.n_mats * self.d * self.f

    def weight_bytes(self) -> int:
        es = 4 if self.dtype == "f32" else 2
        return self.E * self.n_mats * self.d * self.f * es

    def ffn_bytes(self) -> int:
        """HBM bytes the grouped expert FFN must move at least (both GEMM launches): every
        expert's weights once, the P permuted rows read, H [P, f] written and read back, and the
        P output rows written."""
        es = 4 if self.dtype == "f32" else 2
        return self.weight_bytes() + self.P * (2 * self.d + 2 * self.f) * es

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: micro f32, Mixtral shape, many small experts, Switch top-1, decode shape.
WORKLOADS: dict[str, Workload] = {
    "micro": Workload("micro", T=256, d=128, f=512, E=8, k=2, act=ACT_GELU_TANH,
                      gate=GATE_RENORM, dtype="f32", has_bias=True, router_bias_var=None, seed=1),
    "mixtral": Workload("mixtral", T=4096, d=4096, f=14336, E=8, k=2, act=ACT_SWIGLU,
                        gate=GATE_RENORM, dtype="bf16", has_bias=False, router_bias_var=None,
                        seed=2),
    "many_small": Workload("many_small", T=16384, d=2048, f=1408, E=64, k=4, act=ACT_SWIGLU,
                           gate=GATE_RENORM, dtype="bf16", has_bias=False, router_bias_var=2.0,
                           seed=3),
    "switch": Workload("switch", T=32768, d=1024, f=4096, E=128, k=1, act=ACT_GELU_TANH,
                       gate=GATE_RAW_PROB, dtype="bf16", has_bias=False, router_bias_var=None,
                       seed=4),
    # Seed 5 routes at least one token to every expert (checked by the oracle tests), so every
    # forward streams all eight experts' weights.
    "decode": Workload("decode", T=32, d=4096, f=14336, E=8, k=2, act=ACT_SWIGLU,
                       gate=GATE_RENORM, dtype="bf16", has_bias=False, router_bias_var=None,
                       seed=5),
}


def _randn(g: torch.Generator, shape, std: float, dtype: torch.dtype) -> torch.Tensor:
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x if dtype == torch.float32 else x.to(dtype)


def generate(w: Workload, pin_memory: bool = False) -> dict[str, torch.Tensor | None]:
    """Draw every input of workload ``w`` on the host (CPU tensors, contiguous)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    dt = w.torch_dtype
    out: dict[str, torch.Tensor | None] = {}
    out["h"] = _randn(g, (w.T, w.d), 1.0, dt)
    out["W_r"] = _randn(g, (w.d, w.E), 1.0 / math.sqrt(w.d), torch.float32)
    out["b_r"] = (_randn(g, (w.E,), math.sqrt(w.router_bias_var), torch.float32)
                  if w.router_bias_var is not None else None)
    W1 = torch.empty((w.E, w.f, w.d), dtype=dt, pin_memory=pin_memory)
    W3 = torch.empty((w.E, w.f, w.d), dtype=dt, pin_memory=pin_memory) if w.act == ACT_SWIGLU else None
    W2 = torch.empty((w.E, w.d, w.f), dtype=dt, pin_memory=pin_memory)
    s1 = 1.0 / math.sqrt(w.d)
    s2 = 1.0 / math.sqrt(w.f)
    for e in range(w.E):
        W1[e] = _randn(g, (w.f, w.d), s1, dt)
        if W3 is not None:
            W3[e] = _randn(g, (w.f, w.d), s1, dt)
        W2[e] = _randn(g, (w.d, w.f), s2, dt)
    out["W1"], out["W3"], out["W2"] = W1, W3, W2
    out["b1"] = torch.zeros((w.E, w.f), dtype=torch.float32) if w.has_bias else None
    out["b2"] = torch.zeros((w.E, w.d), dtype=torch.float32) if w.has_bias else None
    # drawn last, so that every other input is the same with or without it
    out["sel_bias"] = (_randn(g, (w.E,), w.sel_bias_std, torch.float32)
                       if w.sel_bias_std > 0 else None)
    if pin_memory:
        out["h"] = out["h"].pin_memory()
    return out


def generate_router_inputs(w: Workload) -> dict[str, torch.Tensor | None]:
    """Only h, W_r and b_r of workload ``w``: the first draws of the stream, identical to the ones
    ``generate`` returns, without drawing the expert weights."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    h = _randn(g, (w.T, w.d), 1.0, w.torch_dtype)
    W_r = _randn(g, (w.d, w.E), 1.0 / math.sqrt(w.d), torch.float32)
    b_r = (_randn(g, (w.E,), math.sqrt(w.router_bias_var), torch.float32)
           if w.router_bias_var is not None else None)
    return {"h": h, "W_r": W_r, "b_r": b_r}


def small(name: str = "small", *, T: int, d: int, f: int, E: int, k: int, act: str = ACT_SWIGLU,
          gate: str = GATE_RENORM, dtype: str = "bf16", has_bias: bool = False,
          router_bias_var: float | None = None, seed: int = 11,
          capacity_factor: float = 0.0, fuse_gather: bool = False,
          sel_bias_std: float = 0.0) -> Workload:
    """A custom-shaped workload for parity cases (ragged tails, several tiles, edge cases)."""
    return Workload(name, T=T, d=d, f=f, E=E, k=k, act=act, gate=gate, dtype=dtype,
                    has_bias=has_bias, router_bias_var=router_bias_var, seed=seed,
                    capacity_factor=capacity_factor, fuse_gather=fuse_gather,
                    sel_bias_std=sel_bias_std)


def random_biases(w: Workload, inputs: dict, seed: int) -> dict:
    """Replace the zero expert biases with N(0, 0.1^2) draws, so a parity case exercises them."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = dict(inputs)
    out["b1"] = torch.randn((w.E, w.f), generator=g) * 0.1
    out["b2"] = torch.randn((w.E, w.d), generator=g) * 0.1
    return out
