"""Seeded synthetic workloads for the Muon optimizer step.

This module is shared by the tests, the benchmark and the smoke check.  It
holds parameter shape lists and seeded random-number recipes only: none of
the optimizer's arithmetic lives here, so both the CUDA path and the CPU
oracle can draw their inputs from it without sharing any method code.

Workload shapes follow the HyperParallel FSDP Muon RFC (mindspore
hyper-parallel issue "HyperParallel FSDP Muon优化器性能优化 RFC"):
  * section 3 (Newton-Schulz matrix fusion) names 74 parameters of shape
    [24, 10240] and 3D stacks such as [32, 24, 10240];
  * section 2 (expert slicing) names 3D expert tensors [E, M, N].
The dense-transformer and MoE layer sets are the stated workloads of this
library's benchmark configurations.

Value recipe (every tensor drawn independently):
  * parameters  W ~ N(0, 0.02^2)             seed 1
  * gradients   G ~ N(0, std^2)              seed 0 + step
  * momentum    zero at step 0, fp32
The std of the gradient is 1 for the fp32 correctness case, 1e-2 for the
skinny and MoE sets and 1e-3 for the dense layer set.  A parameter's tensor
is drawn from its own generator seeded with ``seed * 1_000_003 + index`` so
that any single parameter can be regenerated on its own.
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence, Tuple

import torch

__all__ = [
    "Workload", "WORKLOADS", "workload", "param_seed", "draw",
    "make_params", "make_grads", "make_momentum",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    """A list of parameter shapes plus the hyper-parameters of the step."""
    name: str
    shapes: Tuple[Tuple[int, ...], ...]
    dtype: torch.dtype
    grad_std: float
    steps: int = 1
    lr: float = 0.02
    beta: float = 0.95
    wd: float = 0.1
    nesterov: bool = True
    ns_steps: int = 5
    coeffs: Tuple[float, float, float] = (3.4445, -4.7750, 2.0315)
    param_std: float = 0.02

    @property
    def num_slices(self) -> int:
        return sum(s[0] if len(s) == 3 else 1 for s in self.shapes)

    @property
    def num_elements(self) -> int:
        tot = 0
        for s in self.shapes:
            n = 1
            for d in s:
                n *= d
            tot += n
        return tot


def _dense_layers(layers: int) -> Tuple[Tuple[int, ...], ...]:
    out: List[Tuple[int, ...]] = []
    for _ in range(layers):
        out += [(4096, 4096)] * 4
        out += [(11008, 4096)]
        out += [(4096, 11008)] * 2
    return tuple(out)


def _moe_layers(layers: int) -> Tuple[Tuple[int, ...], ...]:
    out: List[Tuple[int, ...]] = []
    for _ in range(layers):
        out += [(2048, 2048)] * 4
        # gate and up projections [E, 1408, 2048], down projection [E, 2048, 1408]
        out += [(16, 1408, 2048)] * 2
        out += [(16, 2048, 1408)]
    out += [(24, 10240)] * 74
    return tuple(out)


WORKLOADS = {
    # one fp32 matrix, grad ~ N(0, 1), a single step
    "fp32_24x1024": Workload(
        "fp32_24x1024", ((24, 1024),), torch.float32, grad_std=1.0, steps=1),
    # 74 separate [24, 10240] bf16 parameters grouped into one [74, 24, 10240] batch
    "skinny_74x24x10240": Workload(
        "skinny_74x24x10240", ((24, 10240),) * 74, torch.bfloat16,
        grad_std=1e-2, steps=10),
    # 8 stacks [32, 24, 10240] plus expert tensors: gate/up [64, 1408, 2048],
    # down [64, 2048, 1408] (the transposed case)
    "stacks_experts": Workload(
        "stacks_experts",
        ((32, 24, 10240),) * 8 + ((64, 1408, 2048),) * 2 + ((64, 2048, 1408),),
        torch.bfloat16, grad_std=1e-2),
    # 24 dense transformer layers
    "dense_24L": Workload(
        "dense_24L", _dense_layers(24), torch.bfloat16, grad_std=1e-3),
    # synthetic MoE model, about 3.7 B parameters
    "moe_24L": Workload(
        "moe_24L", _moe_layers(24), torch.bfloat16, grad_std=1e-2),
    # one layer of the dense set: the 4096-class products at a size for
    # kernel profiles (about 4 GB on the device with its workspace)
    "dense_1L": Workload(
        "dense_1L", _dense_layers(1), torch.bfloat16, grad_std=1e-3),
    # one expert stack of the MoE model: the small dense case used for
    # kernel profiles (about 1.2 GB on the device with its workspace)
    "experts_16x1408x2048": Workload(
        "experts_16x1408x2048", ((16, 1408, 2048),), torch.bfloat16, grad_std=1e-2),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def param_seed(seed: int, index: int) -> int:
    return seed * 1_000_003 + index


def draw(shape: Sequence[int], std: float, seed: int, dtype: torch.dtype,
         device="cpu") -> torch.Tensor:
    """N(0, std^2) samples, drawn in fp32 from a generator on ``device``,
    then rounded (round-to-nearest-even) to ``dtype``."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    x.mul_(std)
    return x.to(dtype)


def make_params(w: Workload, device="cpu", seed: int = 1) -> List[torch.Tensor]:
    return [draw(s, w.param_std, param_seed(seed, i), w.dtype, device)
            for i, s in enumerate(w.shapes)]


def make_grads(w: Workload, step: int = 0, device="cpu", seed: int = 0) -> List[torch.Tensor]:
    return [draw(s, w.grad_std, param_seed(seed + step, i), w.dtype, device)
            for i, s in enumerate(w.shapes)]


def make_momentum(w: Workload, device="cpu") -> List[torch.Tensor]:
    return [torch.zeros(s, dtype=torch.float32, device=device) for s in w.shapes]
