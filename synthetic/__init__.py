"""Seeded synthetic layers for the AWQ scale search.

This module only draws random numbers; it holds none of the method's
arithmetic.  Both the oracle tests and the CUDA path take their inputs from
here, so the two sides always see the same values.

Recipe (one ``torch.Generator`` on the CPU, seeded; every draw in fp32, then
scaled and cast to the layer's dtype):

* W ~ N(0, w_std), shape (out, in).  A shared-input layer group (q/k/v)
  draws each member separately and concatenates them along the output rows.
* X ~ N(0, 1), shape (N, in).
* Outlier input channels: ``randperm(in)[:k]``; every selected column of X is
  multiplied by one factor, either a constant (6, as in the notebook layer of
  "GPTQ and AWQ weight quantisation", section "Setup") or one draw from
  U(20, 100) per channel (the 20x-100x outlier size quoted in "Advanced
  Quantization Algorithms: AWQ and GPTQ Explained", section 1).
* k is the outlier fraction times ``in``, rounded to the nearest integer.

The pages' real workloads are trained LLM layers and calibration text; those
weights and datasets are not available, so these layers stand in for them,
shape for shape.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

import torch

__all__ = ["LayerConfig", "CONFIGS", "make_layer", "make_random_layer", "config_by_name"]


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    out: int
    in_: int
    N: int
    dtype: str          # "f32" | "f16" | "bf16"
    w_std: float
    bits: int
    group: int
    sym: bool
    grid: int           # number of alpha values is grid + 1
    n_outlier: int
    outlier: Tuple      # ("const", factor) or ("uniform", lo, hi)
    n_members: int = 1  # >1: shared-input group, members concatenated row-wise

    @property
    def n_alpha(self) -> int:
        return self.grid + 1

    @property
    def search_flops(self) -> float:
        """Algorithmic flops of the error GEMMs: 2*N*in*out per alpha."""
        return 2.0 * self.N * self.in_ * self.out * self.n_alpha


_TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

CONFIGS = [
    # 128x256 fp32 layer, N=64, 4 channels x6; symmetric 4-bit, group 128.
    LayerConfig("tiny-128x256-n64", 128, 256, 64, "f32", 0.02, 4, 128, True, 20, 4, ("const", 6.0)),
    # 4096x4096 fp16 notebook layer, N=256, 64 channels x6; symmetric 4-bit, group 128.
    LayerConfig("nb-4096x4096-n256", 4096, 4096, 256, "f16", 0.02, 4, 128, True, 20, 64, ("const", 6.0)),
    # 11008x4096 bf16 MLP up projection, N=512, 1% channels x U(20,100); asymmetric 4-bit.
    LayerConfig("up-11008x4096-n512", 11008, 4096, 512, "bf16", 0.02, 4, 128, False, 20, 41,
                ("uniform", 20.0, 100.0)),
    # q/k/v group: three 4096x4096 bf16 layers sharing X, N=2048, 0.5% channels; asymmetric 4-bit.
    LayerConfig("qkv-12288x4096-n2048", 12288, 4096, 2048, "bf16", 0.02, 4, 128, False, 20, 20,
                ("uniform", 20.0, 100.0), n_members=3),
    # 8192x28672 bf16 MLP down projection, N=1024, 0.1% channels; asymmetric 4-bit, 41 alphas.
    LayerConfig("down-8192x28672-n1024", 8192, 28672, 1024, "bf16", 0.01, 4, 128, False, 40, 29,
                ("uniform", 20.0, 100.0)),
]


def config_by_name(name: str) -> LayerConfig:
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)


def _draw(cfg_out: int, in_: int, N: int, dtype: str, w_std: float, n_outlier: int, outlier,
          n_members: int, gen: torch.Generator) -> Tuple[torch.Tensor, torch.Tensor]:
    rows = cfg_out // n_members
    ws = []
    for _ in range(n_members):
        ws.append(torch.randn(rows, in_, generator=gen, dtype=torch.float32) * w_std)
    W = torch.cat(ws, 0) if n_members > 1 else ws[0]
    X = torch.randn(N, in_, generator=gen, dtype=torch.float32)
    if n_outlier > 0:
        ch = torch.randperm(in_, generator=gen)[:n_outlier]
        if outlier[0] == "const":
            X[:, ch] *= float(outlier[1])
        else:
            f = torch.empty(n_outlier, dtype=torch.float32).uniform_(outlier[1], outlier[2], generator=gen)
            X[:, ch] *= f[None, :]
    tdt = _TORCH_DT[dtype]
    return W.to(tdt).contiguous(), X.to(tdt).contiguous()


def make_layer(cfg: LayerConfig, seed: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """(W, X) CPU tensors of the config's dtype, drawn with ``seed``."""
    gen = torch.Generator().manual_seed(seed)
    return _draw(cfg.out, cfg.in_, cfg.N, cfg.dtype, cfg.w_std, cfg.n_outlier, cfg.outlier,
                 cfg.n_members, gen)


def make_random_layer(out: int, in_: int, N: int, dtype: str = "bf16", seed: int = 0,
                      w_std: float = 0.02, n_outlier: Optional[int] = None,
                      outlier=("uniform", 20.0, 100.0)) -> Tuple[torch.Tensor, torch.Tensor]:
    """A small seeded layer of any shape (for parity cases and edge cases)."""
    if n_outlier is None:
        n_outlier = max(1, in_ // 100)
    n_outlier = min(n_outlier, in_)
    gen = torch.Generator().manual_seed(seed)
    return _draw(out, in_, N, dtype, w_std, n_outlier, outlier, 1, gen)
