"""Seeded synthetic GEMM operands.

This module only draws numbers and stores them in the requested operand layout.  It
holds none of the GEMM arithmetic, so both the CUDA path and the CPU checker can take
their inputs from it.

Generation recipe (the same for every problem):
  * one ``torch.Generator('cpu')`` seeded with the problem's seed;
  * draw the LOGICAL A (M x K), then the logical B (K x N), then C (M x N) if present,
    in float32: ``int2`` = integers uniform in {-2..2}; ``uniform`` = U[-1, 1];
    ``normal`` = N(0, sigma) with sigma the standard deviation;
  * cast once to fp16/bf16 (round to nearest even), or, for FP8 inputs (a_fmt / b_fmt
    "e4m3" / "e5m2"), cast A and B once to that format with torch's conversion and keep
    their one-byte codes (C stays in the 16-bit dtype);
  * block-scaled FP8 problems then draw E8M0 scale codes, uniform integers in
    ``scale_codes`` = (lo, hi): SFA (M x ceil(K/32)) and then SFB (N x ceil(K/32)), row-major;
  * store in the requested major.  The values never depend on the major:
      A K-major : A[m*lda + k]      A M-major : A[m + k*lda]
      B K-major : B[n*ldb + k]      B N-major : B[k*ldb + n]
      C, D      : row-major, leading dimension N.

The named workloads are the five GEMM problems the throughput and parity runs use.
"""
from dataclasses import dataclass, replace
from typing import Optional

import torch

K_MAJOR = "K"
MN_MAJOR = "MN"


@dataclass(frozen=True)
class Problem:
    name: str
    M: int
    N: int
    K: int
    dtype: str = "f16"          # "f16" | "bf16": inputs, C and D
    majorA: str = K_MAJOR
    majorB: str = K_MAJOR
    has_c: bool = False
    alpha: float = 1.0
    beta: float = 0.0
    dist: str = "uniform"       # distribution of A and B
    sigma: float = 1.0
    c_dist: str = "normal"
    c_sigma: float = 1.0
    seed: int = 0
    lda: Optional[int] = None   # None = packed
    ldb: Optional[int] = None
    a_fmt: Optional[str] = None  # None: A in dtype; "e4m3" | "e5m2": one-byte FP8 codes
    b_fmt: Optional[str] = None
    scale_codes: Optional[tuple] = None   # block-scaled FP8: E8M0 codes drawn from [lo, hi]

    @property
    def in_bytes(self) -> int:
        return 1 if self.a_fmt else 2

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> int:
        """A, B (input element size), (C) read once and D written once (2 bytes each)."""
        cd = self.M * self.N * (2 if self.has_c else 1)
        return self.in_bytes * (self.M * self.K + self.K * self.N) + 2 * cd

    def with_(self, **kw) -> "Problem":
        return replace(self, **kw)


WORKLOADS = {
    "gemm256_int_f16": Problem("gemm256_int_f16", 256, 256, 256, "f16", dist="int2", seed=0),
    "gemm4096_f16": Problem("gemm4096_f16", 4096, 4096, 4096, "f16", dist="uniform", seed=1),
    "gemm8192_bf16_c": Problem("gemm8192_bf16_c", 8192, 8192, 8192, "bf16", has_c=True,
                               alpha=1.25, beta=0.5, dist="normal", sigma=1.0,
                               c_dist="normal", c_sigma=1.0, seed=2),
    "gemm16384x1024x4096_mnmajor_f16": Problem("gemm16384x1024x4096_mnmajor_f16", 16384,
                                               1024, 4096, "f16", majorA=MN_MAJOR,
                                               majorB=MN_MAJOR, dist="uniform", seed=3),
    "gemm5000x3000x4104_ragged_f16": Problem("gemm5000x3000x4104_ragged_f16", 5000, 3000,
                                             4104, "f16", has_c=True, alpha=0.75, beta=1.0,
                                             dist="uniform", c_dist="normal", c_sigma=0.5,
                                             seed=4),
}
WORKLOAD_ORDER = list(WORKLOADS)

# FP8-input problems: E4M3 x E4M3 with bf16 C and D, the square size of the 16-bit headline.
FP8_WORKLOADS = {
    "gemm8192_e4m3_bf16_c": Problem("gemm8192_e4m3_bf16_c", 8192, 8192, 8192, "bf16",
                                    has_c=True, alpha=1.25, beta=0.5, dist="normal",
                                    sigma=1.0, c_dist="normal", c_sigma=1.0, seed=5,
                                    a_fmt="e4m3", b_fmt="e4m3"),
}
# Block-scaled (MX) FP8: the same square problem with one E8M0 scale per 32 K elements,
# scales between 2^-4 and 2^4.
FP8_WORKLOADS["gemm8192_mxfp8_bf16_c"] = Problem("gemm8192_mxfp8_bf16_c", 8192, 8192, 8192, "bf16",
                                                 has_c=True, alpha=1.25, beta=0.5, dist="normal",
                                                 sigma=1.0, c_dist="normal", c_sigma=1.0, seed=6,
                                                 a_fmt="e4m3", b_fmt="e4m3", scale_codes=(123, 131))
FP8_TORCH = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}

# A decode-like problem with few output tiles (N = 16): K is split across CTAs (stream-K,
# through a workspace) so that every SM has work.  Bound by reading A from HBM.
EXTRA_WORKLOADS = {
    "gemm4096x16x4096_decode_bf16": Problem("gemm4096x16x4096_decode_bf16", 4096, 16, 4096, "bf16",
                                            dist="normal", sigma=1.0, seed=7),
    # the 8192^3 size in fp16 without C (alpha 1, beta 0): the fp16 -> fp32 GEMM the headline
    # metric names, beside the 8192^3 bf16 problem with C that the throughput runs use
    "gemm8192_f16": Problem("gemm8192_f16", 8192, 8192, 8192, "f16", dist="uniform", seed=8),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f16": torch.float16, "bf16": torch.bfloat16}[name]


def _draw(g, shape, dist, sigma):
    if dist == "int2":
        return torch.randint(-2, 3, shape, generator=g).to(torch.float32)
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32) * sigma
    if dist == "ones":
        return torch.ones(shape, dtype=torch.float32)
    raise ValueError(dist)


def _cast(x, dt, fmt):
    if fmt is None:
        return x.to(dt)
    return x.to(FP8_TORCH[fmt]).view(torch.uint8)


def leading_dims(p: Problem):
    lda = p.lda if p.lda is not None else (p.K if p.majorA == K_MAJOR else p.M)
    ldb = p.ldb if p.ldb is not None else (p.K if p.majorB == K_MAJOR else p.N)
    return lda, ldb


def store_a(a_logical: torch.Tensor, major: str, lda: int) -> torch.Tensor:
    """Lay out a logical M x K matrix in its stored form (flat, 1-D)."""
    M, K = a_logical.shape
    if major == K_MAJOR:
        buf = torch.zeros((max(M, 1), lda), dtype=a_logical.dtype)
        buf[:M, :K] = a_logical
    else:
        buf = torch.zeros((max(K, 1), lda), dtype=a_logical.dtype)
        buf[:K, :M] = a_logical.t()
    return buf.reshape(-1)


def store_b(b_logical: torch.Tensor, major: str, ldb: int) -> torch.Tensor:
    """Lay out a logical K x N matrix in its stored form (flat, 1-D)."""
    K, N = b_logical.shape
    if major == K_MAJOR:
        buf = torch.zeros((max(N, 1), ldb), dtype=b_logical.dtype)
        buf[:N, :K] = b_logical.t()
    else:
        buf = torch.zeros((max(K, 1), ldb), dtype=b_logical.dtype)
        buf[:K, :N] = b_logical
    return buf.reshape(-1)


def make(p: Problem, logical: bool = False):
    """Host (CPU) operands for problem p.

    Returns a dict with A, B (flat stored 16-bit tensors, or uint8 FP8 codes), lda, ldb, C
    (flat M*N, or None) and, with logical=True, the logical matrices a (M x K), b (K x N),
    c (M x N).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(p.seed)
    dt = torch_dtype(p.dtype)
    if (p.a_fmt or p.b_fmt) and (p.majorA != K_MAJOR or p.majorB != K_MAJOR):
        raise ValueError("FP8 operands are K-major")
    a = _cast(_draw(g, (p.M, p.K), p.dist, p.sigma), dt, p.a_fmt)
    b = _cast(_draw(g, (p.K, p.N), p.dist, p.sigma), dt, p.b_fmt)
    c = _draw(g, (p.M, p.N), p.c_dist, p.c_sigma).to(dt) if p.has_c else None
    lda, ldb = leading_dims(p)
    out = {
        "A": store_a(a, p.majorA, lda),
        "B": store_b(b, p.majorB, ldb),
        "lda": lda,
        "ldb": ldb,
        "C": c.reshape(-1).clone() if c is not None else None,
    }
    if p.scale_codes is not None:
        lo, hi = p.scale_codes
        nsf = -(-p.K // 32)
        out["SFA"] = torch.randint(lo, hi + 1, (p.M, nsf), generator=g).to(torch.uint8).reshape(-1)
        out["SFB"] = torch.randint(lo, hi + 1, (p.N, nsf), generator=g).to(torch.uint8).reshape(-1)
        out["ld_sf"] = nsf
    if logical:
        out.update(a=a, b=b, c=c)
    return out


def bits(t: torch.Tensor):
    """Raw codes of a CPU tensor as a numpy uint16 array: the 16-bit patterns of fp16/bf16,
    or one-byte FP8 codes (uint8 / float8) widened to 16 bits."""
    import numpy as np
    t = t.contiguous()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy().astype(np.uint16)
    return t.view(torch.int16).numpy().view(np.uint16)
