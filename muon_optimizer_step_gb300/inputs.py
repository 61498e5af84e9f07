"""Seeded synthetic workloads for the Muon step: shapes, hyper-parameters, inputs.

This module holds no arithmetic of the optimizer itself; it only draws the weights,
gradients and (zero) momentum that both the CUDA path and the fp64 oracle consume.
The pages name no dataset, so every workload here is synthetic:

* weights ~ N(0, 0.02^2);
* a gradient for optimizer step t, per matrix of shape r x c, is
  N(0, (1e-3)^2) noise plus a low-rank part P Q^T (P: r x k, Q: c x k standard
  normal) rescaled to Frobenius norm 0.1 * sqrt(r*c / 32768), drawn afresh for every t;
  for the mixture-of-experts set each expert's three gradients are multiplied by
  exp(z_e), z_e ~ N(0, 1) (a lognormal scale with sigma = 1);
* non-matrix parameters get N(0, (1e-3)^2) gradients;
* momentum starts at zero.

Small workloads are drawn on the host with numpy (PCG64 seeded with [seed, stream]).
The multi-gigabyte ones are drawn on the GPU with a seeded torch CUDA generator; the
oracle then checks copies of sampled matrices taken from those same tensors.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

WEIGHT_STD = 0.02
GRAD_NOISE_STD = 1e-3
LOWRANK_NORM_AT_32768 = 0.1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shapes: tuple            # ((rows, cols), ...) in flat-buffer order
    is_matrix: tuple         # bool per parameter
    n_shards: int
    seed: int
    rank: int                # rank of the structured gradient part
    expert_groups: tuple = ()  # ((first param index, count), ...) sharing one lognormal scale
    lr: float = 0.02
    wd: float = 0.01
    mu: float = 0.95
    nesterov: bool = True
    ns_steps: int = 5
    opt_steps: int = 3

    @property
    def numel(self) -> int:
        return sum(r * c for r, c in self.shapes)

    @property
    def n_matrices(self) -> int:
        return sum(1 for f in self.is_matrix if f)

    def matrix_indices(self):
        return [i for i, f in enumerate(self.is_matrix) if f]


def _mats(shapes):
    return tuple((int(r), int(c)) for r, c in shapes)


_GPT2_LAYER = ((768, 2304), (768, 768), (768, 3072), (3072, 768))
_LLAMA_LAYER = ((4096, 4096), (4096, 4096), (1024, 4096), (1024, 4096),
                (14336, 4096), (14336, 4096), (4096, 14336))  # q, o, k, v, gate, up, down
_MOE_EXPERT = ((2048, 1408), (2048, 1408), (1408, 2048))      # gate, up, down


def _workloads():
    w = {}
    w["single_256x128"] = Workload(
        "single_256x128", _mats([(256, 128)]), (True,), 1, seed=0, rank=4)
    sh = _GPT2_LAYER * 12
    w["gpt2_small_x12"] = Workload("gpt2_small_x12", _mats(sh), (True,) * len(sh), 1,
                                   seed=1, rank=8)
    sh = _LLAMA_LAYER * 32
    w["llama3_8b_x32"] = Workload("llama3_8b_x32", _mats(sh), (True,) * len(sh), 1,
                                  seed=2, rank=16)
    sh = _MOE_EXPERT * 64 + ((2048, 2048),) * 4
    groups = tuple((3 * e, 3) for e in range(64))
    w["moe_64e"] = Workload("moe_64e", _mats(sh), (True,) * len(sh), 1, seed=3, rank=8,
                            expert_groups=groups)
    sh = _LLAMA_LAYER * 2
    w["llama3_8b_x2"] = Workload("llama3_8b_x2", _mats(sh), (True,) * len(sh), 1, seed=6,
                                 rank=16)
    sh = ((4096, 1),) + _LLAMA_LAYER * 32
    w["llama3_8b_8shards"] = Workload("llama3_8b_8shards", _mats(sh),
                                      (False,) + (True,) * (len(sh) - 1), 8, seed=4, rank=16)
    # Small parity cases: several 128-wide tiles plus ragged tails, odd shapes,
    # a vector (non-matrix) parameter, a 1 x n row and a 1 x 1 matrix.
    sh = ((300, 200), (37, 1), (130, 520), (200, 200), (1, 50), (7, 3), (64, 1000),
          (257, 129), (1, 1), (384, 256))
    w["ragged_small"] = Workload("ragged_small", _mats(sh),
                                 (True, False, True, True, True, True, True, True, True, True),
                                 3, seed=5, rank=4)
    return w


WORKLOADS = _workloads()


def lowrank_norm(rows, cols):
    return LOWRANK_NORM_AT_32768 * math.sqrt(rows * cols / 32768.0)


# ----------------------------------------------------------------------------- host (numpy)
def host_weights(wl: Workload) -> np.ndarray:
    rng = np.random.default_rng([wl.seed, 0])
    return rng.normal(0.0, WEIGHT_STD, wl.numel).astype(np.float32)


def host_grads(wl: Workload, step: int) -> np.ndarray:
    """Flat fp32 gradient for optimizer step ``step`` (0-based)."""
    rng = np.random.default_rng([wl.seed, 1 + step])
    out = np.empty(wl.numel, dtype=np.float32)
    scales = _expert_scales_host(wl, step)
    pos = 0
    for i, (r, c) in enumerate(wl.shapes):
        n = r * c
        g = rng.normal(0.0, GRAD_NOISE_STD, n)
        if wl.is_matrix[i]:
            k = wl.rank
            P = rng.normal(size=(r, k))
            Q = rng.normal(size=(c, k))
            Lm = P @ Q.T
            nrm = float(np.linalg.norm(Lm))
            if nrm > 0:
                Lm *= lowrank_norm(r, c) / nrm
            g = g + Lm.reshape(-1)
            g *= scales[i]
        out[pos:pos + n] = g
        pos += n
    return out


def _expert_scales_host(wl: Workload, step: int):
    scales = [1.0] * len(wl.shapes)
    if wl.expert_groups:
        rng = np.random.default_rng([wl.seed, 1000 + step])
        z = rng.normal(size=len(wl.expert_groups))
        for (first, count), ze in zip(wl.expert_groups, z):
            for j in range(first, first + count):
                scales[j] = math.exp(float(ze))
    return scales


def host_inputs(wl: Workload):
    """(W0, [G_0, ..., G_{opt_steps-1}], M0) as flat fp32 numpy vectors."""
    W = host_weights(wl)
    Gs = [host_grads(wl, t) for t in range(wl.opt_steps)]
    M = np.zeros(wl.numel, dtype=np.float32)
    return W, Gs, M


# ----------------------------------------------------------------------------- device (torch)
def device_fill_weights(wl: Workload, W, gen_seed_offset: int = 0):
    """Fill a flat fp32 CUDA tensor with N(0, 0.02^2) weights from a seeded generator."""
    import torch
    g = torch.Generator(device=W.device)
    g.manual_seed(wl.seed * 1_000_003 + 17 + gen_seed_offset)
    W.normal_(0.0, WEIGHT_STD, generator=g)


def device_fill_grads(wl: Workload, G, step: int):
    """Fill a flat fp32 CUDA tensor with the step-``step`` gradient of ``wl``."""
    import torch
    g = torch.Generator(device=G.device)
    g.manual_seed(wl.seed * 1_000_003 + 1000 + step)
    G.normal_(0.0, GRAD_NOISE_STD, generator=g)
    zs = None
    if wl.expert_groups:
        zs = torch.randn(len(wl.expert_groups), generator=g, device=G.device,
                         dtype=torch.float64).exp().tolist()
    scales = [1.0] * len(wl.shapes)
    if zs is not None:
        for (first, count), s in zip(wl.expert_groups, zs):
            for j in range(first, first + count):
                scales[j] = s
    prev_tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        pos = 0
        for i, (r, c) in enumerate(wl.shapes):
            n = r * c
            if wl.is_matrix[i]:
                view = G[pos:pos + n].view(r, c)
                P = torch.randn(r, wl.rank, generator=g, device=G.device)
                Q = torch.randn(c, wl.rank, generator=g, device=G.device)
                Lm = P @ Q.T
                nrm = float(torch.linalg.vector_norm(Lm))
                if nrm > 0:
                    Lm.mul_(lowrank_norm(r, c) / nrm)
                view.add_(Lm)
                if scales[i] != 1.0:
                    view.mul_(scales[i])
                del Lm, P, Q
            pos += n
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev_tf32
