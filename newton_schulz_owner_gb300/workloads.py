"""Seeded synthetic workloads: projection-set shapes and input tensors.

This module holds no arithmetic of the Muon step.  It only lists parameter
shapes and draws seeded random inputs, so that the CUDA library's tests, the
benchmark and the fp64 oracle's tests can all be fed identical data.

The model shapes are those of the pages' LLM runs (DMuon home page,
"LLM Pretraining" and the "Benchmarks" table: Qwen2.5 1.5B-7B and Llama-3
3B-8B).  No checkpoint is read: every tensor is drawn from a seeded normal
distribution; real weights and gradients are not needed to exercise the step.
Shapes are PyTorch ``(out, in)``, row-major and contiguous.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import torch

Shape = Tuple[int, int]

# Per-layer projection order: q, k, v, o, gate, up, down.
_PROJ_ORDER = ("q", "k", "v", "o", "gate", "up", "down")


def _layer(hidden: int, kv: int, ffn: int) -> Dict[str, Shape]:
    return {"q": (hidden, hidden), "k": (kv, hidden), "v": (kv, hidden),
            "o": (hidden, hidden), "gate": (ffn, hidden), "up": (ffn, hidden),
            "down": (hidden, ffn)}


@dataclass(frozen=True)
class Workload:
    """A named projection set plus the distributions its inputs are drawn from."""
    name: str
    index: int                       # used in the per-matrix seed 1000*index + i
    layers: int
    layer_shapes: Dict[str, Shape] = field(default_factory=dict)
    grad_dtype: torch.dtype = torch.bfloat16
    weight_dtype: torch.dtype = torch.bfloat16
    grad_std: float = 1e-3
    weight_std: float = 0.02
    n_owners: int = 1
    vocab: int = 0                   # embedding rows (0: no AdamW parameters)
    tied_head: bool = False          # output head shares the embedding

    def shapes(self) -> List[Shape]:
        out: List[Shape] = []
        for _ in range(self.layers):
            for p in _PROJ_ORDER:
                if p in self.layer_shapes:
                    out.append(self.layer_shapes[p])
        return out

    def adamw_shapes(self) -> List[Shape]:
        """Parameters outside the Muon set, updated by AdamW: token embedding,
        output head (when not tied to the embedding), and the RMSNorm weights
        (two per layer plus the final one), as (rows, cols)."""
        if self.vocab <= 0:
            return []
        hidden = self.layer_shapes["q"][1]
        out = [(self.vocab, hidden)]
        if not self.tied_head:
            out.append((self.vocab, hidden))
        out += [(1, hidden)] * (2 * self.layers + 1)
        return out

    def names(self) -> List[str]:
        out: List[str] = []
        for l in range(self.layers):
            for p in _PROJ_ORDER:
                if p in self.layer_shapes:
                    out.append(f"layers.{l}.{p}_proj")
        return out


WORKLOADS: Dict[str, Workload] = {
    # One 256x1024 fp32 gradient N(0,1), zero momentum, fp32 weight N(0, 0.02^2).
    "single-256x1024": Workload("single-256x1024", 0, 1, {"q": (256, 1024)},
                                grad_dtype=torch.float32, weight_dtype=torch.float32,
                                grad_std=1.0, weight_std=0.02),
    "qwen2.5-1.5b": Workload("qwen2.5-1.5b", 1, 28, _layer(1536, 256, 8960),
                             vocab=151936, tied_head=True),
    "llama-3.2-3b": Workload("llama-3.2-3b", 2, 28, _layer(3072, 1024, 8192), n_owners=8,
                             vocab=128256, tied_head=True),
    "llama-3.1-8b": Workload("llama-3.1-8b", 3, 32, _layer(4096, 1024, 14336), vocab=128256),
    "qwen2.5-7b": Workload("qwen2.5-7b", 4, 28, _layer(3584, 512, 18944), vocab=152064),
    # One layer of the Llama-3.1-8B set (7 matrices, 218 M elements, ~3.5 GB on
    # the device with workspace): the same kernels on a case small enough for
    # multi-pass profiler captures.
    "llama-3.1-8b-layer": Workload("llama-3.1-8b-layer", 5, 1, _layer(4096, 1024, 14336)),
    # One layer of the Qwen2.5-1.5B set with the model's (tied) embedding as its
    # AdamW parameters (233 M elements, ~4 GB on the device in all): the AdamW
    # kernel on a case small enough for multi-pass profiler captures.
    "qwen2.5-1.5b-layer": Workload("qwen2.5-1.5b-layer", 6, 1, _layer(1536, 256, 8960),
                                   vocab=151936, tied_head=True),
}


def seed_for(workload: Workload, i: int, step: int = 0) -> int:
    """Seed of matrix i's gradient at a given step (weights use step = -1)."""
    return 1000 * workload.index + i + 1_000_003 * (step + 1)


def _randn(shape: Shape, seed: int, device: torch.device, std: float,
           dtype: torch.dtype, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    t = t.to(dtype)                  # RNE cast to bf16 when dtype is bf16
    if out is not None:
        out.copy_(t)
        return out
    return t


def _round_up(v: int, a: int) -> int:
    return (v + a - 1) // a * a


@dataclass
class FlatSet:
    """One flat allocation holding every matrix, each segment 256-byte aligned."""
    flat: torch.Tensor
    views: List[torch.Tensor]
    offsets: List[int]


def alloc_flat(shapes: Sequence[Shape], dtype: torch.dtype, device, *, pin: bool = False,
               zero: bool = True) -> FlatSet:
    esz = torch.empty((), dtype=dtype).element_size()
    align = 256 // esz
    offs, cur = [], 0
    for r, c in shapes:
        offs.append(cur)
        cur = _round_up(cur + r * c, align)
    cur = max(cur, align)
    if pin:
        flat = torch.empty(cur, dtype=dtype, pin_memory=True)
        if zero:
            flat.zero_()
    else:
        flat = (torch.zeros if zero else torch.empty)(cur, dtype=dtype, device=device)
    views = [flat[o:o + r * c].view(r, c) for o, (r, c) in zip(offs, shapes)]
    return FlatSet(flat, views, offs)


def fill_grads(workload: Workload, fs: FlatSet, step: int = 0,
               indices: Optional[Sequence[int]] = None) -> None:
    """Draw the step's gradients G_i ~ N(0, grad_std^2) into the flat set."""
    dev = fs.flat.device
    for i in (range(len(fs.views)) if indices is None else indices):
        v = fs.views[i]
        _randn(tuple(v.shape), seed_for(workload, i, step), dev, workload.grad_std,
               v.dtype, out=v)


def fill_weights(workload: Workload, fs: FlatSet,
                 indices: Optional[Sequence[int]] = None) -> None:
    """Draw weights W_i ~ N(0, weight_std^2) into the flat set."""
    dev = fs.flat.device
    for i in (range(len(fs.views)) if indices is None else indices):
        v = fs.views[i]
        _randn(tuple(v.shape), seed_for(workload, i, -1) + 7, dev, workload.weight_std,
               v.dtype, out=v)


def random_matrix(shape: Shape, seed: int, device="cpu", std: float = 1.0,
                  dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """A single seeded N(0, std^2) matrix (used for odd test shapes)."""
    return _randn(tuple(shape), seed, torch.device(device), std, dtype)
