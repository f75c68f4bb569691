"""Seeded synthetic workloads for the NVFP4 block-scaled GEMM.

This module only draws random bytes; it holds none of the GEMM's arithmetic,
so the CUDA path's tests and the CPU oracle can both consume its output.

Distribution (same for every workload unless noted):
  * FP4 operand bytes are uniform over 0..255, i.e. two independent nibbles,
    each uniform over the 16 E2M1 codes; byte i of a row holds k = 2i in its low
    nibble and k = 2i+1 in its high nibble.
  * Scale bytes are E4M3 codes of 2^j * (1 + f/8): the byte is ((j+7) << 3) | f
    with j uniform in [j_lo, j_hi] and f uniform in 0..7.  j in [-4, 1] except
    for the 8192^3 problem, which uses j in [-3, 0].
  * One ``torch.Generator`` seeded once per workload; per group the draws come
    in the order A, SFA, B, SFB.
  * The MoE workload's group sizes are M in {64,128,192,256,384,512,768,1024}
    put in the order of ``torch.randperm(8)`` under seed 0.

Layouts (per group): A [L, M, K/2], B [L, N, K/2], SFA [L, M, K/16],
SFB [L, N, K/16], all uint8, row-major; C is fp16 [L, M, N].
"""
from dataclasses import dataclass, field
from typing import List, Tuple

import torch

MOE_M_SIZES = (64, 128, 192, 256, 384, 512, 768, 1024)


def moe_m_order(seed: int = 0) -> List[int]:
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(len(MOE_M_SIZES), generator=g).tolist()
    return [MOE_M_SIZES[i] for i in perm]


@dataclass
class Workload:
    name: str
    shapes: List[Tuple[int, int, int, int]]  # (M, N, K, L) per group
    j_range: Tuple[int, int] = (-4, 1)
    description: str = ""

    @property
    def flops(self) -> int:
        return sum(2 * M * N * K * L for M, N, K, L in self.shapes)

    @property
    def bytes(self) -> int:
        """Unique operand bytes a GEMM must move: A, B (K/2 per row), SFA, SFB
        (K/16 per row) and C (2 per element)."""
        tot = 0
        for M, N, K, L in self.shapes:
            tot += L * (M * K // 2 + N * K // 2 + M * K // 16 + N * K // 16 + 2 * M * N)
        return tot


WORKLOADS = {
    "single_128x128x256": Workload(
        "single_128x128x256", [(128, 128, 256, 1)],
        description="single NVFP4 GEMM M=128 N=128 K=256"),
    "skinny_128x7168x16384": Workload(
        "skinny_128x7168x16384", [(128, 7168, 16384, 1)],
        description="skinny-M dense NVFP4 GEMM M=128 N=7168 K=16384 (HBM-bound on B)"),
    "dense_8192x8192x8192": Workload(
        "dense_8192x8192x8192", [(8192, 8192, 8192, 1)], j_range=(-3, 0),
        description="compute-bound dense NVFP4 GEMM M=N=K=8192"),
    "grouped2": Workload(
        "grouped2", [(1024, 4096, 7168, 1), (2048, 7168, 2048, 1)],
        description="grouped NVFP4 GEMM, 2 groups (1024x4096x7168, 2048x7168x2048)"),
    "moe8": Workload(
        "moe8", [(m, 4096, 7168, 1) for m in moe_m_order(0)],
        description="MoE grouped NVFP4 GEMM, 8 groups N=4096 K=7168, M in a seed-0 permutation"),
}

# The order the problem statement lists them in.
WORKLOAD_ORDER = ["single_128x128x256", "skinny_128x7168x16384", "dense_8192x8192x8192",
                  "grouped2", "moe8"]


def draw_codes(gen: torch.Generator, L: int, rows: int, K: int) -> torch.Tensor:
    return torch.randint(0, 256, (L, rows, K // 2), dtype=torch.uint8, generator=gen)


def draw_scales(gen: torch.Generator, L: int, rows: int, K: int, j_range=(-4, 1)) -> torch.Tensor:
    shape = (L, rows, K // 16)
    j = torch.randint(j_range[0], j_range[1] + 1, shape, dtype=torch.int32, generator=gen)
    f = torch.randint(0, 8, shape, dtype=torch.int32, generator=gen)
    return (((j + 7) << 3) | f).to(torch.uint8)


def make_problem(gen: torch.Generator, M: int, N: int, K: int, L: int = 1, j_range=(-4, 1)) -> dict:
    A = draw_codes(gen, L, M, K)
    SFA = draw_scales(gen, L, M, K, j_range)
    B = draw_codes(gen, L, N, K)
    SFB = draw_scales(gen, L, N, K, j_range)
    return dict(A=A, SFA=SFA, B=B, SFB=SFB, M=M, N=N, K=K, L=L)


def make_inputs(workload, seed: int = 0) -> List[dict]:
    """All groups of a workload (by name or Workload), CPU uint8 tensors."""
    if isinstance(workload, str):
        workload = WORKLOADS[workload]
    gen = torch.Generator().manual_seed(seed)
    return [make_problem(gen, M, N, K, L, workload.j_range) for (M, N, K, L) in workload.shapes]


def make_random_problem(seed: int, M: int, N: int, K: int, L: int = 1, j_range=(-4, 1)) -> dict:
    gen = torch.Generator().manual_seed(seed)
    return make_problem(gen, M, N, K, L, j_range)
