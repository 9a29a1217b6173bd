"""Seeded synthetic inputs for the allreduce-fusion epilogue.

This module holds no arithmetic of the method: it only draws random numbers
and rounds them to the element type, so that the CUDA path and the CPU oracle
see identical bits.  Both sides import it; it imports neither.

Recipe (one CPU ``torch.Generator`` seeded with ``seed``, draws in this order):
  for each rank r = 0..R-1:
      base_r  = randn(T, H) * p_std
      if heavy_frac > 0:
          u_r  = rand(T, H);  hv_r = randn(T, H) * heavy_std
          base_r[u_r < heavy_frac] = hv_r[u_r < heavy_frac]
      partial_r = base_r rounded (RNE) to D (exact for D = fp32)
  residual = randn(T, H) * x_std  -> D
  gamma    = 1 + randn(H) * g_std  -> D
Plain R-way sum inputs: for each rank, (rand(N) * 2 - 1) -> D, i.e. U(-1, 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# Output pattern names (the four combinations the fused operation supports,
# with the quantised output either FP8 E4M3 or NVFP4).
RES_NORM = "res_norm"
NORM = "norm"
RES_QUANT_FP8 = "res_fp8"
RES_QUANT_NVFP4 = "res_nvfp4"
RES_NORM_FP8 = "res_norm_fp8"
RES_NORM_NVFP4 = "res_norm_nvfp4"


@dataclass(frozen=True)
class FusedWorkload:
    name: str
    R: int
    T: int
    H: int
    dtype: str = "bf16"
    p_std: float = 1.0
    x_std: float = 1.0
    g_std: float = 0.1
    heavy_frac: float = 0.0
    heavy_std: float = 20.0
    eps: float = 1e-6
    pattern: str = RES_NORM
    seed: int = 0

    def with_(self, **kw) -> "FusedWorkload":
        d = dict(self.__dict__)
        d.update(kw)
        return FusedWorkload(**d)


@dataclass(frozen=True)
class SumWorkload:
    name: str
    R: int
    N: int
    dtype: str = "fp16"
    seed: int = 0


# The five target workloads.
TINY = FusedWorkload("r2_t16_h512_res_norm", R=2, T=16, H=512, eps=1e-6, pattern=RES_NORM)
DECODE = FusedWorkload("r8_t128_h4096_res_norm", R=8, T=128, H=4096, p_std=0.5, eps=1e-5,
                       pattern=RES_NORM)
FP8_PREFILL = FusedWorkload("r4_t2048_h8192_res_norm_fp8", R=4, T=2048, H=8192, eps=1e-6,
                            pattern=RES_NORM_FP8)
NVFP4_PREFILL = FusedWorkload("r8_t8192_h7168_res_nvfp4", R=8, T=8192, H=7168,
                              heavy_frac=0.01, heavy_std=20.0, eps=1e-6, pattern=RES_QUANT_NVFP4)
SUM_SIZES = [1024 * 4 ** k for k in range(10)] + [1_000_003]
SUMS = [SumWorkload(f"sum_r8_n{n}", R=8, N=n) for n in SUM_SIZES]

FUSED = [TINY, DECODE, FP8_PREFILL, NVFP4_PREFILL]

# fp32 elements (the 4-byte exchange type of fp32 Lamport workspaces): the
# decode shape above and a prefill-sized row set with NVFP4 output.
FP32_DECODE = FusedWorkload("r8_t128_h4096_fp32_res_norm", R=8, T=128, H=4096, dtype="fp32",
                            p_std=0.5, eps=1e-5, pattern=RES_NORM)
FP32_PREFILL = FusedWorkload("r8_t1024_h7168_fp32_res_norm_nvfp4", R=8, T=1024, H=7168,
                             dtype="fp32", heavy_frac=0.01, eps=1e-6, pattern=RES_NORM_NVFP4)


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[name]


@dataclass
class FusedInputs:
    partials: torch.Tensor   # [R, T, H] D, CPU
    residual: torch.Tensor   # [T, H] D, CPU
    gamma: torch.Tensor      # [H] D, CPU
    eps: float
    extra: dict = field(default_factory=dict)


def make_fused_inputs(w: FusedWorkload) -> FusedInputs:
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    dt = torch_dtype(w.dtype)
    partials = torch.empty((w.R, w.T, w.H), dtype=dt)
    for r in range(w.R):
        base = torch.randn((w.T, w.H), generator=g, dtype=torch.float32)
        base.mul_(w.p_std)
        if w.heavy_frac > 0:
            u = torch.rand((w.T, w.H), generator=g, dtype=torch.float32)
            hv = torch.randn((w.T, w.H), generator=g, dtype=torch.float32)
            hv.mul_(w.heavy_std)
            m = u < w.heavy_frac
            base[m] = hv[m]
            del u, hv, m
        partials[r].copy_(base)
        del base
    residual = (torch.randn((w.T, w.H), generator=g, dtype=torch.float32) * w.x_std).to(dt)
    gamma = (1.0 + torch.randn((w.H,), generator=g, dtype=torch.float32) * w.g_std).to(dt)
    return FusedInputs(partials, residual, gamma, w.eps)


def make_sum_inputs(w: SumWorkload, device: str = "cpu") -> torch.Tensor:
    """[R, N] inputs, each rank (rand(N) * 2 - 1) -> D.  ``device`` picks where
    the seeded generator runs: the CPU stream (default, what parity tests
    use) or a device generator (same recipe and distribution, another stream;
    for inputs too large to draw on the host quickly)."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    dt = torch_dtype(w.dtype)
    out = torch.empty((w.R, w.N), dtype=dt, device=device)
    for r in range(w.R):
        out[r].copy_(torch.rand((w.N,), generator=g, dtype=torch.float32, device=device)
                     .mul_(2.0).sub_(1.0))
    return out


def bits(t: torch.Tensor):
    """CPU float tensor -> numpy bit patterns (uint16 for 16-bit types, uint32
    for fp32; no copy of values through any float conversion)."""
    import numpy as np
    if t.element_size() == 4:
        return t.contiguous().view(torch.int32).numpy().view(np.uint32)
    assert t.element_size() == 2
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a, dtype: str) -> torch.Tensor:
    import numpy as np
    if dtype == "fp32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).view(
            torch.float32)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(
        torch_dtype(dtype))
