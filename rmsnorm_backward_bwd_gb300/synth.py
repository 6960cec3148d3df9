"""Seeded synthetic inputs and the workload table.

This module holds no RMSNorm arithmetic: it only draws random tensors and
names the shapes that tests and the benchmark run. Both the CUDA path and the
CPU oracle receive the very same tensors from here.

Recipe: one ``torch.Generator`` on the CPU, seeded (default 0), draws fp32
standard normals in the fixed order x, residual (fused-add only), gamma, dy,
dresidual_out (fused-add with a residual gradient only); then
gamma = 1 + 0.1 * N(0,1), dy and dresidual_out are scaled by their workload's
factor, and every tensor is cast to the I/O dtype (round to nearest even).
The distributions follow the shapes and value ranges the FlyDSL pages test
(f32 / f16 / bf16, aligned and unaligned N, N <= 2048, M up to LLM training
sizes); the pages use no public dataset.
"""
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclass(frozen=True)
class Case:
    """One backward problem: shape, dtype, which variant, value scales."""
    name: str
    M: int
    N: int
    dtype: str
    fused: bool = False
    with_dres: bool = False
    eps: float = 1e-6
    dy_scale: float = 0.01
    dres_scale: float = 0.01
    seed: int = 0


def make_inputs(case: Case, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Draw the case's tensors in the fixed order; return them in case.dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(case.seed)
    M, N = case.M, case.N
    f32 = torch.float32
    out = {}
    out["x"] = torch.randn(M, N, generator=g, dtype=f32)
    if case.fused:
        out["residual"] = torch.randn(M, N, generator=g, dtype=f32)
    out["gamma"] = 1.0 + 0.1 * torch.randn(N, generator=g, dtype=f32)
    out["dy"] = torch.randn(M, N, generator=g, dtype=f32) * case.dy_scale
    if case.fused and case.with_dres:
        out["dres"] = torch.randn(M, N, generator=g, dtype=f32) * case.dres_scale
    dt = TORCH_DTYPES[case.dtype]
    return {k: v.to(dt).to(device) for k, v in out.items()}


def make_ln_inputs(case: Case, x_shift: float = 0.5, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """LayerNorm inputs: one CPU generator seeded with case.seed draws fp32
    normals in the order x, gamma, dy, beta; x is shifted by x_shift (rows
    with a nonzero mean, so that the centring matters), gamma = 1 + 0.1*N(0,1),
    dy is scaled by case.dy_scale, beta = 0.1*N(0,1); all cast to the dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(case.seed)
    M, N = case.M, case.N
    f32 = torch.float32
    out = {}
    out["x"] = torch.randn(M, N, generator=g, dtype=f32) + x_shift
    out["gamma"] = 1.0 + 0.1 * torch.randn(N, generator=g, dtype=f32)
    out["dy"] = torch.randn(M, N, generator=g, dtype=f32) * case.dy_scale
    out["beta"] = 0.1 * torch.randn(N, generator=g, dtype=f32)
    dt = TORCH_DTYPES[case.dtype]
    return {k: v.to(dt).to(device) for k, v in out.items()}


def ln_algorithmic_bytes(M: int, N: int, dtype: str, with_dbeta: bool, casts: bool) -> int:
    """Bytes a LayerNorm backward call must move: read x, dy, gamma, mean and
    rstd; write dx, dgamma_f32 [and dbeta_f32], and the casts when requested
    and dtype != f32."""
    s = ELEM_BYTES[dtype]
    nout = 2 if with_dbeta else 1
    b = M * N * s * 3 + N * s + 8 * M + 4 * N * nout
    if casts and dtype != "f32":
        b += N * s * nout
    return b


def algorithmic_bytes(M: int, N: int, dtype: str, with_dres: bool, dweight_cast: bool) -> int:
    """Bytes a backward call must move: read x|added, dy, [dres], gamma, rstd;
    write dx, dweight_f32 and (when requested and dtype != f32) the cast dweight."""
    s = ELEM_BYTES[dtype]
    b = M * N * s * (4 if with_dres else 3) + N * s + 4 * M + 4 * N
    if dweight_cast and dtype != "f32":
        b += N * s
    return b


# The workloads: the small fwd+bwd check, the two 4096x4096 bf16 backwards,
# the edge-shape sweep and the large training shape.
SMALL_F32 = Case("rmsnorm fwd+bwd f32 M=128 N=1024", 128, 1024, "f32", eps=1e-5, dy_scale=1.0)
PLAIN_4096 = Case("rmsnorm_bwd bf16 M=4096 N=4096", 4096, 4096, "bf16")
FUSED_4096 = Case("fused_add_rmsnorm_bwd bf16 M=4096 N=4096 +dres", 4096, 4096, "bf16",
                  fused=True, with_dres=True)
FUSED_4096_NODRES = Case("fused_add_rmsnorm_bwd bf16 M=4096 N=4096 dres=None", 4096, 4096,
                         "bf16", fused=True, with_dres=False)
EDGE_SHAPES = [(1, 4096, "bf16"), (512, 2048, "bf16"), (512, 3000, "f32"), (128, 4096, "f16")]
LARGE_PLAIN = Case("rmsnorm_bwd bf16 M=16384 N=8192", 16384, 8192, "bf16")
LARGE_FUSED = Case("fused_add_rmsnorm_bwd bf16 M=16384 N=8192 +dres", 16384, 8192, "bf16",
                   fused=True, with_dres=True)


LN_4096 = Case("layernorm_bwd bf16 M=4096 N=4096", 4096, 4096, "bf16", eps=1e-5)
LN_LARGE = Case("layernorm_bwd bf16 M=16384 N=8192", 16384, 8192, "bf16", eps=1e-5)
# rows that are not 16-byte multiples (the staged phase-class kernel, one team of 512 threads)
LN_UNALIGNED = Case("layernorm_bwd bf16 M=4096 N=8190", 4096, 8190, "bf16", eps=1e-5)
# rows longer than one CTA's tile (the cluster engine's range)
LONG_ROWS = Case("rmsnorm_bwd bf16 M=4096 N=32768", 4096, 32768, "bf16")
# rows that are not 16-byte multiples (the generic engines' range: phase-class kernel)
UNALIGNED_ROWS = Case("rmsnorm_bwd bf16 M=4096 N=4095", 4096, 4095, "bf16")
# rows of 24 KB that are not 16-byte multiples (phase-class kernel, four chunks a thread)
UNALIGNED_WIDE_ROWS = Case("rmsnorm_bwd bf16 M=4096 N=12290", 4096, 12290, "bf16")


def edge_cases() -> List[Case]:
    cases = []
    for M, N, dt in EDGE_SHAPES:
        cases.append(Case("rmsnorm_bwd %s M=%d N=%d" % (dt, M, N), M, N, dt))
        cases.append(Case("fused_add_rmsnorm_bwd %s M=%d N=%d +dres" % (dt, M, N), M, N, dt,
                          fused=True, with_dres=True))
    return cases
