"""Seeded synthetic inputs for the ZeRO flat-parameter step.

This module is the only code shared by the CUDA path's tests/benchmark and
the oracle: it describes workloads (parameter lists of the model layouts and
how they group into FlatParameter units) and draws seeded random values.  It
contains none of the method's arithmetic (no padding, reduction, Adam or
rounding of results).

Value recipe (every draw is seeded):
  * fp32 initial parameters ~ N(0, 0.02)
  * replica gradients ~ N(0, sigma), stored as bf16 (torch's round-to-nearest
    conversion of the fp32 draw) or as fp32; optional outliers: a seeded
    fraction of positions set to +-1.
Large buffers are drawn directly on the device that will hold them with a
seeded ``torch.Generator``; the oracle reads back exactly those bytes.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Sequence

import numpy as np
import torch


# ---------------------------------------------------------------------------
# Workload layouts: ordered parameter lists and their unit (FlatParameter) ids.
# ---------------------------------------------------------------------------
@dataclass
class ParamList:
    name: str
    numel: List[int] = field(default_factory=list)
    unit: List[int] = field(default_factory=list)
    names: List[str] = field(default_factory=list)

    def add(self, name: str, numel: int, unit: int) -> None:
        self.names.append(name)
        self.numel.append(int(numel))
        self.unit.append(int(unit))

    @property
    def total(self) -> int:
        return int(sum(self.numel))

    @property
    def n_units(self) -> int:
        return (max(self.unit) + 1) if self.unit else 0


def mlp_params(widths: Sequence[int], name: str = "mlp") -> ParamList:
    """One FlatParameter per Linear layer (W then b), layer i = unit i."""
    pl = ParamList(name)
    for i in range(len(widths) - 1):
        pl.add(f"layer{i}.weight", widths[i] * widths[i + 1], i)
        pl.add(f"layer{i}.bias", widths[i + 1], i)
    return pl


def llama_params(hidden: int, intermediate: int, heads: int, kv_heads: int, layers: int,
                 vocab: int, *, embed: bool = True, head: bool = True, final_norm: bool = True,
                 unit_per_layer: bool = True, name: str = "llama") -> ParamList:
    """Llama-style decoder parameters in module order (untied embeddings).

    Order: embed_tokens; per layer q, k, v, o, gate, up, down, input_norm,
    post_attention_norm; final norm; lm_head.  With ``unit_per_layer`` the
    embedding is unit 0, each decoder layer its own unit, and final norm +
    lm_head share the last unit; otherwise everything is unit 0.
    """
    head_dim = hidden // heads
    kv = kv_heads * head_dim
    pl = ParamList(name)
    u = 0
    if embed:
        pl.add("embed_tokens", vocab * hidden, u)
        if unit_per_layer:
            u += 1
    for layer in range(layers):
        p = f"layers.{layer}."
        pl.add(p + "q_proj", hidden * hidden, u)
        pl.add(p + "k_proj", hidden * kv, u)
        pl.add(p + "v_proj", hidden * kv, u)
        pl.add(p + "o_proj", hidden * hidden, u)
        pl.add(p + "gate_proj", hidden * intermediate, u)
        pl.add(p + "up_proj", hidden * intermediate, u)
        pl.add(p + "down_proj", intermediate * hidden, u)
        pl.add(p + "input_layernorm", hidden, u)
        pl.add(p + "post_attention_layernorm", hidden, u)
        if unit_per_layer:
            u += 1
    if final_norm:
        pl.add("norm", hidden, u)
    if head:
        pl.add("lm_head", vocab * hidden, u)
    return pl


def single_buffer(numel: int, name: str = "flat") -> ParamList:
    pl = ParamList(name)
    pl.add("flat", numel, 0)
    return pl


def from_units(unit_sizes: Sequence[int], name: str = "units") -> ParamList:
    pl = ParamList(name)
    for i, s in enumerate(unit_sizes):
        pl.add(f"unit{i}", s, i)
    return pl


# The workloads the method is exercised on (sizes of the model families).
def toy_mlp() -> ParamList:
    """5-layer MLP, Linear widths 32-128-128-64-64-16 (34,192 params)."""
    return mlp_params([32, 128, 128, 64, 64, 16], "toy_mlp_32-128-128-64-64-16")


def lecture_mlp() -> ParamList:
    """The lecture's zero.py MLP: units of 3168, 9312, 9312, 9312, 1552 (widths 32-96x4-16)."""
    return mlp_params([32, 96, 96, 96, 96, 16], "lecture_mlp_32-96-96-96-96-16")


def llama_1024() -> ParamList:
    """hidden 1024, intermediate 2048, 16/4 heads, 8 layers, vocab 1024, one flat unit."""
    return llama_params(1024, 2048, 16, 4, 8, 1024, unit_per_layer=False, name="llama_h1024_L8_v1024")


def llama_2048_units() -> ParamList:
    """hidden 2048, intermediate 8192, 32/8 heads, 8 layers, vocab 40960, unit per layer."""
    return llama_params(2048, 8192, 32, 8, 8, 40960, unit_per_layer=True, name="llama_h2048_L8_v40960")


def llama_2048_stage_buffer() -> ParamList:
    """32 decoder layers + input embedding of the 2048/8192 model, one flat unit."""
    return llama_params(2048, 8192, 32, 8, 32, 40960, head=False, final_norm=False,
                        unit_per_layer=False, name="llama_h2048_L32_stage")


# ---------------------------------------------------------------------------
# Seeded values.
# ---------------------------------------------------------------------------
def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_fp32(n: int, std: float, seed: int, device="cpu") -> torch.Tensor:
    """n fp32 values ~ N(0, std), drawn on ``device``."""
    out = torch.empty(int(n), dtype=torch.float32, device=device)
    if n:
        out.normal_(0.0, std, generator=_gen(seed, device))
    return out


def replica_grads(n_ranks: int, n: int, std: float, seed: int, dtype: str = "bf16",
                  device="cpu", outlier_fraction: float = 0.0, pad_from: int | None = None
                  ) -> List[torch.Tensor]:
    """N replica gradient buffers of n elements, replica r seeded (seed, r).

    ``outlier_fraction``: that fraction of positions (seeded) is set to +-1.
    ``pad_from``: entries from this index on are zero (the zero pad the
    ZeRO-2 hook appends before the reduce-scatter).
    """
    out = []
    for r in range(n_ranks):
        g = normal_fp32(n, std, seed * 1009 + r, device)
        if outlier_fraction > 0.0 and n > 0:
            k = max(1, int(round(outlier_fraction * n)))
            gen = _gen(seed * 7919 + r, device)
            pos = torch.randint(0, n, (k,), generator=gen, device=device)
            sign = torch.randint(0, 2, (k,), generator=gen, device=device).to(torch.float32) * 2 - 1
            g[pos] = sign
        if pad_from is not None:
            g[pad_from:] = 0
        out.append(g.to(torch.bfloat16) if dtype == "bf16" else g)
    return out


def unit_grads_from_flat(flat: torch.Tensor, bases: Sequence[int], sizes: Sequence[int]):
    """Views of a flat gradient buffer per unit."""
    return [flat[b:b + s] for b, s in zip(bases, sizes)]


def as_numpy_bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy; bf16 tensors come back as their uint16 bit patterns."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()
