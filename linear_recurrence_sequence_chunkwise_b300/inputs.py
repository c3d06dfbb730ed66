"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the retention method: it only draws seeded
Gaussian tensors, rounds them to the storage dtype and names the workloads.
Both the GPU side and the oracle receive exactly the tensors made here (the
oracle widens the stored bf16/fp32 values to fp64 exactly).

Workloads (sizes follow the RetNet pages' setting of multi-scale heads with a
fixed per-head decay; the pages give no benchmark data, so every input is
synthetic):
  tiny            b1  H2  dk16  dv16  N64     chunk 16   fp32  N(0,1)
  parallel_norm   b8  H8  dk256 dv512 N2048              bf16  N(0,1), G N(0,1)
  chunkwise_long  b1  H16 dk256 dv512 N32768  chunk 256  bf16  N(0,1)/sqrt(dk)
  sweep           b4  H16 dk256 dv512 N in {2048,8192,16384} x chunk in {64,128,256}
  decode          b128 H16 dk256 dv512, state N(0, sigma=0.1), 512 steps of
                  bf16 q,k,v ~ N(0,1)/sqrt(dk)
  backward        b4  H16 dk256 dv512 N2048   chunk 64   bf16 q,k,v,dout N(0,1)/sqrt(dk)
  rglru           b8  T4096 D4096 (RG-LRU scan)          bf16 x, gate pre-activations N(0,1),
                  Lambda with a^8 ~ U(0.9, 0.999)
Decay schedule: gamma_h = 1 - 2^(-5-h) (one fixed decay per head, as the
multi-scale retention section prescribes; the schedule itself is a choice).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


def gammas(H: int) -> list[float]:
    """Per-head decays 1 - 2^(-5-h), exactly representable in fp64."""
    return [1.0 - 2.0 ** (-5 - h) for h in range(H)]


@dataclass(frozen=True)
class Workload:
    name: str
    b: int
    H: int
    N: int
    dk: int
    dv: int
    dtype: str            # storage dtype of q, k, v: "f32" or "bf16"
    scale: float          # standard deviation of q, k, v
    chunk: int = 0        # chunk length B for the chunkwise form (0: not used)
    flags: int = 0        # score normalisation flags for the parallel form
    eps: float = 1e-5     # GroupNorm eps for the epilogue
    steps: int = 0        # decode steps
    state_std: float = 0.0
    seed: int = 0
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def gamma(self) -> list[float]:
        return gammas(self.H)


NORM_ALL = 1 | 2 | 4

TINY = Workload("tiny", 1, 2, 64, 16, 16, "f32", 1.0, chunk=16, seed=1000)
PARALLEL_NORM = Workload("parallel_norm", 8, 8, 2048, 256, 512, "bf16", 1.0,
                         flags=NORM_ALL, eps=1e-5, seed=2000)
CHUNKWISE_LONG = Workload("chunkwise_long", 1, 16, 32768, 256, 512, "bf16", 1.0 / 16.0,
                          chunk=256, seed=3000)
SWEEP = [Workload(f"sweep_N{N}_B{B}", 4, 16, N, 256, 512, "bf16", 1.0 / 16.0, chunk=B,
                  seed=4000 + 10 * i + j)
         for i, N in enumerate((2048, 8192, 16384)) for j, B in enumerate((64, 128, 256))]
DECODE = Workload("decode", 128, 16, 1, 256, 512, "bf16", 1.0 / 16.0, steps=512,
                  state_std=0.1, seed=5000)

# gradient of the chunkwise form at the first training-sweep shape; dout ~ N(0,1)/sqrt(dk)
BACKWARD = Workload("backward", 4, 16, 2048, 256, 512, "bf16", 1.0 / 16.0, chunk=64, seed=6000)

# RG-LRU scan (Griffin page): b rows, T steps, D channels; x and the two gate
# pre-activations N(0,1) bf16, Lambda drawn so that a^c is uniform in [0.9, 0.999] (the
# page's initialisation), zero initial state, fp32 output.  Workload fields: N = T,
# dv = D (dk unused).
RGLRU = Workload("rglru", 8, 1, 4096, 0, 4096, "bf16", 1.0, seed=7000)

WORKLOADS = {w.name: w for w in [TINY, PARALLEL_NORM, CHUNKWISE_LONG, DECODE, BACKWARD,
                                 RGLRU] + SWEEP}

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def randn(shape, seed: int, std: float = 1.0, dtype: str = "f32", device="cpu") -> torch.Tensor:
    """Seeded N(0, std^2) tensor rounded (round-to-nearest-even) to ``dtype``.

    On the CPU the stream is numpy's PCG64 (stable across versions); on a CUDA
    device it is torch's Philox generator.  Callers that compare against the
    oracle always hand it the very tensor they used, so the two streams never
    need to agree with each other.
    """
    device = torch.device(device)
    shape = tuple(int(s) for s in shape)
    if device.type == "cpu":
        rng = np.random.Generator(np.random.PCG64(seed))
        t = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32))
    else:
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(_TORCH_DTYPE[dtype])


def qkv(w: Workload, device="cpu", N: int | None = None, seed_offset: int = 0):
    """Q, K, V of a workload: q,k [b,H,N,dk], v [b,H,N,dv] in the storage dtype."""
    N = w.N if N is None else N
    s = w.seed + seed_offset
    q = randn((w.b, w.H, N, w.dk), s + 1, w.scale, w.dtype, device)
    k = randn((w.b, w.H, N, w.dk), s + 2, w.scale, w.dtype, device)
    v = randn((w.b, w.H, N, w.dv), s + 3, w.scale, w.dtype, device)
    return q, k, v


def dout(w: Workload, device="cpu", N: int | None = None) -> torch.Tensor:
    """Upstream gradient of the output, [b,H,N,dv] in the storage dtype."""
    N = w.N if N is None else N
    return randn((w.b, w.H, N, w.dv), w.seed + 7, w.scale, w.dtype, device)


def rglru_lambda(D: int, seed: int, c: float = 8.0, device="cpu") -> torch.Tensor:
    """Lambda [D] fp32 with a^c ~ U(0.9, 0.999) for a = sigmoid(Lambda), the Griffin page's
    initialisation: a = u^(1/c), Lambda = log(a / (1 - a)) (computed in fp64)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.uniform(0.9, 0.999, size=D) ** (1.0 / c)
    return torch.from_numpy(np.log(a / (1.0 - a))).to(torch.float32).to(device)


def rglru_inputs(w: Workload, device="cpu", T: int | None = None):
    """x, gate_a, gate_x [b,T,D] in the storage dtype and Lambda [D] fp32."""
    T = w.N if T is None else T
    shape = (w.b, T, w.dv)
    x = randn(shape, w.seed + 1, w.scale, w.dtype, device)
    ga = randn(shape, w.seed + 2, 1.0, w.dtype, device)
    gx = randn(shape, w.seed + 3, 1.0, w.dtype, device)
    return x, ga, gx, rglru_lambda(w.dv, w.seed + 4, 8.0, device)


def gate(w: Workload, device="cpu", N: int | None = None) -> torch.Tensor:
    """The swish gate input G = X W_G, token-major [b, N, H*dv], bf16 N(0,1)."""
    N = w.N if N is None else N
    return randn((w.b, N, w.H * w.dv), w.seed + 4, 1.0, "bf16", device)


def decode_state(w: Workload, device="cpu") -> torch.Tensor:
    """Initial decode state S_0 [b,H,dk,dv], fp32 N(0, state_std^2)."""
    return randn((w.b, w.H, w.dk, w.dv), w.seed + 5, w.state_std, "f32", device)


def decode_step_inputs(w: Workload, step: int, device="cpu"):
    """q, k [b,H,dk] and v [b,H,dv] of one decode step (bf16)."""
    s = w.seed + 100 + 3 * step
    q = randn((w.b, w.H, w.dk), s, w.scale, w.dtype, device)
    k = randn((w.b, w.H, w.dk), s + 1, w.scale, w.dtype, device)
    v = randn((w.b, w.H, w.dv), s + 2, w.scale, w.dtype, device)
    return q, k, v


def decode_all_inputs(w: Workload, device="cpu"):
    """All decode steps at once: q,k [steps,b,H,dk], v [steps,b,H,dv] (bf16)."""
    q = randn((w.steps, w.b, w.H, w.dk), w.seed + 101, w.scale, w.dtype, device)
    k = randn((w.steps, w.b, w.H, w.dk), w.seed + 102, w.scale, w.dtype, device)
    v = randn((w.steps, w.b, w.H, w.dv), w.seed + 103, w.scale, w.dtype, device)
    return q, k, v


def algorithmic_flops(kind: str, w: Workload, N: int | None = None) -> float:
    """Useful flop count of one call (2 flop per multiply-add, causal half only).

    parallel:  per head, the causal QK^T and score x V products:
               (dk + dv) * N * (N + 1)
    chunkwise: per token per head, intra-chunk causal part (dk+dv)(B+1) plus the
               cross-chunk read and the state update, 2*dk*dv each.
    decode:    per (b,h) per step: state update 2*dk*dv, read-out 2*dk*dv.
    backward:  per token per head, three causal intra-chunk parts (dq, dk, dv)
               3 (dk+dv)(B+1), three cross-chunk reads 6*dk*dv and two carried
               states (the forward one for dq, the gradient one shared by dk and dv)
               4*dk*dv.
    """
    N = w.N if N is None else N
    if kind == "parallel":
        return float(w.b * w.H) * (w.dk + w.dv) * N * (N + 1)
    if kind == "chunkwise":
        per_tok = (w.dk + w.dv) * (w.chunk + 1) + 4 * w.dk * w.dv
        return float(w.b * w.H) * N * per_tok
    if kind == "decode":
        return float(w.b * w.H) * 4.0 * w.dk * w.dv
    if kind == "backward":
        per_tok = 3 * (w.dk + w.dv) * (w.chunk + 1) + 10 * w.dk * w.dv
        return float(w.b * w.H) * N * per_tok
    raise ValueError(kind)


def esize(dtype: str) -> int:
    return 2 if dtype == "bf16" else 4


def sqrt_dk(w: Workload) -> float:
    return math.sqrt(w.dk)
