"""Seeded synthetic inputs for y = FP16(x . W^T) + b.

The one module that both the CUDA path's tests/benchmark and the oracle's
callers use: it draws numbers and holds none of the method's arithmetic.
Values are drawn in FP32 from a CPU torch.Generator and stored as binary16
(torch's own conversion); the same host tensors feed both sides.

Workloads (shapes and distributions of the linear op studied in "Tensor
Programs, Part 1": the toy linear, plus decode, prefill and MLP projection
shapes with the same [out_features, in_features] weight layout):
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist: str          # "uniform", "smallint" or "normal"
    seed: int
    description: str

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        # x and W read once, b read once, y written once (binary16)
        return 2 * (self.M * self.K + self.N * self.K + self.N + self.M * self.N)


WORKLOADS = {
    w.name: w for w in [
        Workload("toy", 1024, 1024, 768, "uniform", 1000,
                 "toy linear: x [1024,768], W [1024,768], b [1024], U[-1,1]"),
        Workload("ragged_exact", 2047, 1000, 770, "smallint", 1001,
                 "exactness/ragged: small integers in [-4,4], tails in M, N and K"),
        Workload("gemv_m1", 1, 4096, 4096, "normal", 1002, "decode-row GEMV, M=1"),
        Workload("gemv_m8", 8, 4096, 4096, "normal", 1003, "decode-row GEMV, M=8"),
        Workload("prefill", 4096, 4096, 4096, "normal", 1004, "prefill projection 4096^3"),
        Workload("mlp_up", 8192, 14336, 4096, "normal", 1005, "MLP up-projection"),
    ]
}


def make_inputs(M: int, N: int, K: int, dist: str, seed: int):
    """x [M,K], w [N,K], b [N] as contiguous float16 CPU tensors.

    uniform:  x, W, b ~ U[-1, 1]
    smallint: x, W, b integers uniform in [-4, 4]
    normal:   x ~ N(0, 1), W ~ N(0, 0.02^2), b ~ N(0, 0.1^2)  (0.02 and 0.1
              are standard deviations)
    """
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    if dist == "uniform":
        x = torch.rand((M, K), generator=g, dtype=torch.float32) * 2 - 1
        w = torch.rand((N, K), generator=g, dtype=torch.float32) * 2 - 1
        b = torch.rand((N,), generator=g, dtype=torch.float32) * 2 - 1
    elif dist == "smallint":
        x = torch.randint(-4, 5, (M, K), generator=g).to(torch.float32)
        w = torch.randint(-4, 5, (N, K), generator=g).to(torch.float32)
        b = torch.randint(-4, 5, (N,), generator=g).to(torch.float32)
    elif dist == "normal":
        x = torch.randn((M, K), generator=g, dtype=torch.float32)
        w = torch.randn((N, K), generator=g, dtype=torch.float32) * 0.02
        b = torch.randn((N,), generator=g, dtype=torch.float32) * 0.1
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.half().contiguous(), w.half().contiguous(), b.half().contiguous()


def workload_inputs(name: str, seed_offset: int = 0):
    wl = WORKLOADS[name]
    return make_inputs(wl.M, wl.N, wl.K, wl.dist, wl.seed + seed_offset)
