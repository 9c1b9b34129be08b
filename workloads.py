"""Seeded synthetic inputs for the GEMM workloads (shared by tests and bench).

This module holds no GEMM arithmetic: it draws random matrices with a seeded
CPU ``torch.Generator``, rounds them to the input dtype (round-to-nearest-even,
done by torch's casts) and returns the raw bits.  Both the CUDA path and the
oracle consume exactly these bits.

Workloads (stand-ins for the sweeps of "[Persistent] Performance on
09-persistent-matmul on A100 worse than non-persistent": M=N=4K with K from 128
to 4096 step 128 and M=N=8K with K from 256 to 8192 step 256, both fp16; plus a
square fp16 case, an fp8 case and tail-effect shapes):

  fp16_512          M=N=K=512, A,B ~ U[-1, 1], fp16 in, fp16 out
  fp16_4096_ksweep  M=N=4096, K=128..4096 step 128, A,B ~ N(0,1)/sqrt(K)
  bf16_8192_ksweep  M=N=8192, K=256..8192 step 256, A,B ~ N(0,1)/sqrt(K)
  e4m3_8192         M=N=K=8192, A,B ~ N(0,1), scaled per tensor so max|x| = 448,
                    rounded to e4m3; C in bf16 with the dequant scale applied
  bf16_tail         (5120,5120,4096), (4224,3968,2048), (19200,256,8192)
  bf16_grouped_vark 64 problems of M=N=1024 in one grouped launch, K log-uniform
                    in [256, 8192] (multiples of 8), A,B ~ N(0,1)/sqrt(K): tiles
                    whose cost varies 32-fold, where a dynamic scheduler can
                    balance what a static one cannot

A is M x K row-major; B is stored N x K row-major (K x N column-major).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

F16, BF16, E4M3 = 0, 1, 2
DTYPE_NAMES = {F16: "f16", BF16: "bf16", E4M3: "e4m3"}
E4M3_MAX = 448.0


@dataclass(frozen=True)
class Problem:
    name: str
    M: int
    N: int
    K: int
    dtype: int
    dist: str        # "uniform" (U[-1,1]) | "normal_sqrtk" (N(0,1)/sqrt(K)) | "normal" (N(0,1))
    seed: int


def fp16_512() -> List[Problem]:
    return [Problem("fp16_512", 512, 512, 512, F16, "uniform", 1000)]


def fp16_4096_ksweep(ks: Optional[List[int]] = None) -> List[Problem]:
    ks = ks or list(range(128, 4096 + 1, 128))
    return [Problem(f"fp16_4096_k{k}", 4096, 4096, k, F16, "normal_sqrtk", 2000 + k) for k in ks]


def bf16_8192_ksweep(ks: Optional[List[int]] = None) -> List[Problem]:
    ks = ks or list(range(256, 8192 + 1, 256))
    return [Problem(f"bf16_8192_k{k}", 8192, 8192, k, BF16, "normal_sqrtk", 3000 + k) for k in ks]


def e4m3_8192() -> List[Problem]:
    return [Problem("e4m3_8192", 8192, 8192, 8192, E4M3, "normal", 4000)]


def bf16_tail() -> List[Problem]:
    shapes = [(5120, 5120, 4096), (4224, 3968, 2048), (19200, 256, 8192)]
    return [Problem(f"bf16_tail_{m}x{n}x{k}", m, n, k, BF16, "normal_sqrtk", 5000 + i)
            for i, (m, n, k) in enumerate(shapes)]


def bf16_grouped_vark(count: int = 64, M: int = 1024, N: int = 1024, seed: int = 6000) -> List[Problem]:
    """`count` bf16 problems of M x N whose K differ: K = 8 * round(2^u / 8)
    with u ~ U[8, 13] drawn by a generator seeded `seed` (problem i's inputs
    are seeded seed + 1 + i)."""
    gen = torch.Generator().manual_seed(seed)
    u = torch.rand(count, generator=gen, dtype=torch.float64) * 5.0 + 8.0
    ks = [max(8, 8 * int(round(2.0 ** float(x) / 8.0))) for x in u]
    return [Problem(f"bf16_grouped_{i}_{M}x{N}x{k}", M, N, k, BF16, "normal_sqrtk", seed + 1 + i)
            for i, k in enumerate(ks)]


WORKLOADS = {
    "fp16_512": fp16_512,
    "fp16_4096_ksweep": fp16_4096_ksweep,
    "bf16_8192_ksweep": bf16_8192_ksweep,
    "e4m3_8192": e4m3_8192,
    "bf16_tail": bf16_tail,
    "bf16_grouped_vark": bf16_grouped_vark,
}


def _draw(gen: torch.Generator, rows: int, cols: int, dist: str, K: int) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(rows, cols, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    x = torch.randn(rows, cols, generator=gen, dtype=torch.float32)
    if dist == "normal_sqrtk":
        x = x / math.sqrt(max(K, 1))
    elif dist != "normal":
        raise ValueError(dist)
    return x


def _to_e4m3(x: torch.Tensor):
    """Per-tensor scale to max|x| = 448, clamp, round to e4m3 (RNE)."""
    amax = float(x.abs().max()) if x.numel() else 1.0
    scale = np.float32(E4M3_MAX / amax) if amax > 0 else np.float32(1.0)
    y = (x * float(scale)).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return y, float(scale)


@dataclass
class Inputs:
    problem: Problem
    A: torch.Tensor          # CPU tensor in the input dtype (float16 / bfloat16 / float8_e4m3fn)
    B: torch.Tensor          # N x K
    scale_a: float = 1.0
    scale_b: float = 1.0

    def bits(self, which: str) -> np.ndarray:
        t = self.A if which == "A" else self.B
        if t.dtype == torch.float8_e4m3fn:
            return t.view(torch.uint8).numpy()
        return t.view(torch.int16).numpy().view(np.uint16)


def make_inputs(p: Problem) -> Inputs:
    """Draw A (M x K) then B (N x K) from one generator seeded with p.seed."""
    gen = torch.Generator().manual_seed(p.seed)
    a = _draw(gen, p.M, p.K, p.dist, p.K)
    b = _draw(gen, p.N, p.K, p.dist, p.K)
    if p.dtype == E4M3:
        a8, sa = _to_e4m3(a)
        b8, sb = _to_e4m3(b)
        return Inputs(p, a8.contiguous(), b8.contiguous(), sa, sb)
    td = torch.float16 if p.dtype == F16 else torch.bfloat16
    return Inputs(p, a.to(td).contiguous(), b.to(td).contiguous())


def custom(M: int, N: int, K: int, dtype: int, dist: str = "uniform", seed: int = 0) -> Inputs:
    return make_inputs(Problem(f"custom_{M}x{N}x{K}", M, N, K, dtype, dist, seed))


def output_torch_dtype(dtype: int) -> torch.dtype:
    """C is fp16 for fp16 inputs and bf16 for bf16 and e4m3 inputs."""
    return torch.float16 if dtype == F16 else torch.bfloat16
