"""Seeded synthetic inputs for the fused low-rank-adapted linear layer.

This module only draws random numbers and casts them to the storage dtype.  It
holds none of the layer's arithmetic, so both the CPU oracle (``oracle/``) and
the GPU path (``dora_adapter_linear_gb300``) can consume the very same inputs
without sharing any code of the method itself.

Recipe (all on the CPU with ``torch.Generator().manual_seed(seed)``, drawn in
fp32 in a fixed order, then rounded to the storage dtype; the oracle receives
the rounded values upcast to fp64):

* X, dY ~ N(0, 1); W0, A ~ N(0, 1/in); B ~ N(0, 0.02^2); bias ~ N(0, 0.01^2)
* DoRA magnitude m = rownorm(W0) * U(0.9, 1.1) (column variant: colnorm(W0) *
  U(0.9, 1.1), one entry per input feature) -- the workload's own recipe for the
  magnitude vector; it is an input, not part of the forward pass
* dropout keep mask: uint8, 1 with probability 1 - p, drawn as U(0, 1) >= p with its own seed
* W8A8: X and W0 are drawn as above and left unquantised; quantisation is part
  of the method and lives on each side separately.

The pages measure on workloads that are not available here (a shape sweep of
adapter kernels, audio-model and diffusion-model training); these Gaussian
tensors of LLM/DiT projection sizes stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

__all__ = ["LinearCase", "MlpCase", "W8A8Case", "QkvCase", "WORKLOADS", "make_linear", "make_mlp",
           "make_w8a8", "make_qkv", "make_dropout_mask", "scaled"]


@dataclass(frozen=True)
class LinearCase:
    """One LoRA / DoRA linear workload: y = X W0^T + s (X A^T) B^T (+bias)."""
    name: str
    M: int
    d_in: int
    d_out: int
    r: int
    alpha: float
    dtype: str            # "f32" or "bf16"
    dora: bool = False
    dora_cols: bool = False   # DoRA column variant: magnitude per input column
    bias: bool = False
    eps: float = 1e-12
    strength: float = 1.0
    seed: int = 1000

    @property
    def s(self) -> float:
        return self.strength * self.alpha / self.r


@dataclass(frozen=True)
class MlpCase:
    """LoRA SwiGLU MLP: h = silu(X Wg'^T) * (X Wu'^T), y = h Wd'^T.  r is the gate projection's
    rank; r_u and r_d (None: the same as r) those of the up and down projections."""
    name: str
    M: int
    H: int
    I: int
    r: int
    alpha: float
    dtype: str = "bf16"
    seed: int = 1003
    r_u: int = None
    r_d: int = None

    @property
    def ranks(self) -> dict:
        return {"g": self.r, "u": self.r_u or self.r, "d": self.r_d or self.r}

    @property
    def s(self) -> float:
        return self.alpha / self.r

    @property
    def scales(self) -> dict:
        """s = alpha / rank of each projection."""
        return {p: self.alpha / rk for p, rk in self.ranks.items()}


@dataclass(frozen=True)
class W8A8Case:
    """int8 base weight (per-row scales), int8 per-token activations, bf16 LoRA."""
    name: str
    M: int
    d_in: int
    d_out: int
    r: int
    alpha: float
    bias: bool = False
    seed: int = 1004

    @property
    def s(self) -> float:
        return self.alpha / self.r


@dataclass(frozen=True)
class QkvCase:
    """Fused query/key/value projection: W0 [sum n, d_in], one rank-r adapter per leaf."""
    name: str
    M: int
    d_in: int
    n: tuple              # output rows of each leaf
    r: int
    alpha: float
    strengths: tuple = (1.0, 0.75, 1.25)   # per leaf, so that leaf scales are told apart
    bias: bool = False
    seed: int = 1005

    @property
    def s(self) -> tuple:
        return tuple(st * self.alpha / self.r for st in self.strengths[:len(self.n)])


# The workloads, named by what they are.  The tiny fp32 one and the
# reduced ("small") variants are sized so the fp64 oracle finishes in seconds.
WORKLOADS = {
    "lora_tiny_f32": LinearCase("lora_tiny_f32", 64, 256, 256, 8, 8.0, "f32", bias=True, seed=1000),
    "lora_4096_bf16": LinearCase("lora_4096_bf16", 8192, 4096, 4096, 16, 32.0, "bf16", seed=1001),
    "dora_4096x11008_bf16": LinearCase("dora_4096x11008_bf16", 8192, 4096, 11008, 32, 32.0, "bf16",
                                        dora=True, bias=True, seed=1002),
    "dora_cols_4096x11008_bf16": LinearCase("dora_cols_4096x11008_bf16", 8192, 4096, 11008, 32, 32.0, "bf16",
                                             dora_cols=True, bias=True, seed=1006),
    "mlp_swiglu_4096x14336_bf16": MlpCase("mlp_swiglu_4096x14336_bf16", 16384, 4096, 14336, 16, 16.0),
    "w8a8_lora_3072": W8A8Case("w8a8_lora_3072", 16384, 3072, 3072, 32, 32.0),
    # grouped-query attention block of a 4096-wide model: 32 query heads, 8 key/value heads of 128
    "qkv_lora_4096_gqa_bf16": QkvCase("qkv_lora_4096_gqa_bf16", 16384, 4096, (4096, 1024, 1024), 16, 16.0),
}


def scaled(case, **kw):
    """Same workload recipe with some sizes replaced (for small parity cases)."""
    d = dict(case.__dict__)
    d.update(kw)
    return type(case)(**d)


_TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _normal(g, shape, std):
    return torch.randn(*shape, generator=g, dtype=torch.float32) * std


def make_linear(case: LinearCase):
    """Return a dict of CPU tensors in the storage dtype (X, W0, A, B, bias, m, dY)."""
    g = torch.Generator().manual_seed(case.seed)
    dt = _TORCH_DT[case.dtype]
    X = _normal(g, (case.M, case.d_in), 1.0)
    W0 = _normal(g, (case.d_out, case.d_in), case.d_in ** -0.5)
    A = _normal(g, (case.r, case.d_in), case.d_in ** -0.5)
    B = _normal(g, (case.d_out, case.r), 0.02)
    bias = _normal(g, (case.d_out,), 0.01) if case.bias else None
    m_noise = torch.rand(case.d_in if case.dora_cols else case.d_out, generator=g, dtype=torch.float32) * 0.2 + 0.9
    dY = _normal(g, (case.M, case.d_out), 1.0)
    out = {"X": X.to(dt), "W0": W0.to(dt), "A": A.to(dt), "B": B.to(dt), "dY": dY.to(dt),
           "bias": None if bias is None else bias.to(dt)}
    if case.dora or case.dora_cols:
        # magnitude recipe of the workload: row (column, for the column variant) norm of the
        # stored W0 times U(0.9, 1.1)
        w = out["W0"].float()
        out["m"] = (torch.sqrt((w * w).sum(0 if case.dora_cols else 1)) * m_noise).to(dt)
    return out


def make_mlp(case: MlpCase):
    """CPU tensors for the SwiGLU MLP: X, (Wg, Ag, Bg), (Wu, Au, Bu), (Wd, Ad, Bd), dY."""
    g = torch.Generator().manual_seed(case.seed)
    dt = _TORCH_DT[case.dtype]
    H, I = case.H, case.I
    out = {"X": _normal(g, (case.M, H), 1.0).to(dt)}
    for p, (n_out, n_in) in (("g", (I, H)), ("u", (I, H)), ("d", (H, I))):
        r = case.ranks[p]
        out["W" + p] = _normal(g, (n_out, n_in), n_in ** -0.5).to(dt)
        out["A" + p] = _normal(g, (r, n_in), n_in ** -0.5).to(dt)
        out["B" + p] = _normal(g, (n_out, r), 0.02).to(dt)
    out["dY"] = _normal(g, (case.M, H), 1.0).to(dt)
    return out


def make_w8a8(case: W8A8Case):
    """CPU tensors for the W8A8 workload, before quantisation (X bf16, W0 fp32)."""
    g = torch.Generator().manual_seed(case.seed)
    X = _normal(g, (case.M, case.d_in), 1.0).to(torch.bfloat16)
    W0 = _normal(g, (case.d_out, case.d_in), case.d_in ** -0.5)
    A = _normal(g, (case.r, case.d_in), case.d_in ** -0.5).to(torch.bfloat16)
    B = _normal(g, (case.d_out, case.r), 0.02).to(torch.bfloat16)
    bias = _normal(g, (case.d_out,), 0.01).to(torch.bfloat16) if case.bias else None
    return {"X": X, "W0": W0, "A": A, "B": B, "bias": bias}


def make_qkv(case: QkvCase):
    """CPU bf16 tensors for the fused-leaf workload: X, W0, A<l>, B<l> per leaf, bias, dY."""
    g = torch.Generator().manual_seed(case.seed)
    dt = torch.bfloat16
    N = sum(case.n)
    out = {"X": _normal(g, (case.M, case.d_in), 1.0).to(dt),
           "W0": _normal(g, (N, case.d_in), case.d_in ** -0.5).to(dt)}
    for l, nl in enumerate(case.n):
        out[f"A{l}"] = _normal(g, (case.r, case.d_in), case.d_in ** -0.5).to(dt)
        out[f"B{l}"] = _normal(g, (nl, case.r), 0.02).to(dt)
    out["bias"] = _normal(g, (N,), 0.01).to(dt) if case.bias else None
    out["dY"] = _normal(g, (case.M, N), 1.0).to(dt)
    return out


def make_dropout_mask(M: int, d_in: int, p: float, seed: int = 2001):
    """uint8 [M, d_in] keep mask (1 = kept), each entry kept with probability 1 - p."""
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(M, d_in, generator=g, dtype=torch.float32) >= p).to(torch.uint8)
