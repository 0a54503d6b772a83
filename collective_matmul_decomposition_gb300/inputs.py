"""Seeded synthetic inputs for the decomposed collective matmul.

This module is the only code shared between the CUDA path and the fp64
oracle.  It draws random numbers and lays them out; it holds none of the
method's arithmetic (no products, no sums, no schedule).

Shapes follow the Megatron sequence-parallel layers that the AllGather->GEMM
and GEMM->ReduceScatter patterns come from ("Hiding Tensor-Parallel
Collectives: AG/RS Overlap in Megatron", sections 1-5; "Tensor Parallelism ->
Communication Patterns", column/row split):

* AG-GEMM: a global activation X [N*m, K] is sequence-sharded into N row
  shards X_j = X[j*m:(j+1)*m]; a global weight W [K, N*n] is column-split into
  N rank shards W_r = W[:, r*n:(r+1)*n].  Stored as x [N][m][K] and w [N][K][n]
  ("kn", row-major W_r) or w [N][n][K] ("nk", nn.Linear order).
* GEMM-RS: a global activation X [M, N*k] is split along its columns into
  X_r = X[:, r*k:(r+1)*k] and a global weight W [N*k, n] along its rows into
  W_r = W[r*k:(r+1)*k].  Stored as x [N][M][k] and w [N][k][n] or [N][n][k].

Draws are fp32 from a CPU torch.Generator, then rounded to bf16 (round to
nearest even).  uniform[-1,1) is rand*2-1; N(0, s) is randn*s.
"""

from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Dist:
    kind: str  # "uniform" (on [-1, 1)) or "normal"
    std: float = 1.0


UNIFORM = Dist("uniform")
NORMAL1 = Dist("normal", 1.0)
NORMAL002 = Dist("normal", 0.02)


def _draw(shape, dist: Dist, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    if dist.kind == "uniform":
        t = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist.kind == "normal":
        t = torch.randn(shape, generator=g, dtype=torch.float32) * float(dist.std)
    else:
        raise ValueError(f"unknown distribution {dist.kind!r}")
    return t.to(torch.bfloat16)


def _w_layout(w: torch.Tensor, layout: str) -> torch.Tensor:
    """w is [N][K][n]; return it in the requested per-rank layout, contiguous."""
    if layout == "kn":
        return w.contiguous()
    if layout == "nk":
        return w.transpose(1, 2).contiguous()
    raise ValueError(f"unknown weight layout {layout!r}")


def ag_inputs(N: int, m: int, K: int, n: int, x_dist: Dist, w_dist: Dist,
              seed: int, w_layout: str = "nk"):
    """Inputs of AllGather->GEMM: x [N][m][K] bf16 and w per rank (see module doc)."""
    X = _draw((N * m, K), x_dist, seed)              # global, sequence-sharded by rows
    W = _draw((K, N * n), w_dist, seed + 1)          # global, column-split across ranks
    x = X.view(N, m, K)
    w = W.view(K, N, n).permute(1, 0, 2)             # [N][K][n]
    return x.contiguous(), _w_layout(w, w_layout)


def rs_inputs(N: int, M: int, k: int, n: int, x_dist: Dist, w_dist: Dist,
              seed: int, w_layout: str = "nk"):
    """Inputs of GEMM->ReduceScatter: x [N][M][k] bf16 and w per rank (see module doc)."""
    X = _draw((M, N * k), x_dist, seed)              # global, split along the contraction
    W = _draw((N * k, n), w_dist, seed + 1)          # global, split along its rows
    x = X.view(M, N, k).permute(1, 0, 2)             # [N][M][k]
    w = W.view(N, k, n)                              # [N][k][n]
    return x.contiguous(), _w_layout(w, w_layout)


def tagged_ag_inputs(N: int, m: int, K: int, n: int, w_layout: str = "nk"):
    """Placement probe: every output element is an exact small integer.

    X_j[i, 0] = j + 1, X_j[i, 1] = i mod 256, all other entries 0.
    W_r is a 0/1 selector: column c reads input column (c + r) mod 2.
    So Y_r[j*m + i, c] is j+1 or i mod 256, which names the source shard/row.
    Requires K >= 2.
    """
    x = torch.zeros(N, m, K, dtype=torch.float32)
    x[:, :, 0] = (torch.arange(N, dtype=torch.float32) + 1.0).view(N, 1)
    x[:, :, 1] = (torch.arange(m) % 256).to(torch.float32).view(1, m)
    w = torch.zeros(N, K, n, dtype=torch.float32)
    for r in range(N):
        cols = torch.arange(n)
        w[r, (cols + r) % 2, cols] = 1.0
    return x.to(torch.bfloat16).contiguous(), _w_layout(w.to(torch.bfloat16), w_layout)


def int_inputs(shape_x, shape_w, lo: int, hi: int, seed: int):
    """Small-integer bf16 tensors (exact in bf16 for |v| <= 256)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    x = torch.randint(lo, hi + 1, shape_x, generator=g).to(torch.bfloat16)
    w = torch.randint(lo, hi + 1, shape_w, generator=g).to(torch.bfloat16)
    return x.contiguous(), w.contiguous()


def bf16_bits(t: torch.Tensor):
    """The raw uint16 bit patterns of a bf16 CPU tensor, as a numpy array."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# The five workloads, by what they are.  Each entry gives the shapes of both
# operations where the workload has both.
WORKLOADS = {
    "tiny_n2": dict(  # AG and RS at N=2, small enough for the full oracle
        N=2, ag=dict(m=64, K=256, n=512, x=UNIFORM, w=NORMAL002, seed=1000),
        rs=dict(M=128, k=128, n=512, x=UNIFORM, w=NORMAL002, seed=1002),
        y_dtype="f32", direction="uni", chunks=1),
    "sp_mlp_fc1_ag_n8": dict(  # Megatron-SP MLP fc1, seq 4096 / hidden 4096 / ffn shard 2048
        N=8, ag=dict(m=512, K=4096, n=2048, x=NORMAL1, w=NORMAL002, seed=2000),
        y_dtype="bf16", direction="uni", chunks=1),
    "sp_mlp_fc2_rs_n8": dict(  # Megatron-SP MLP fc2, rows 4096, k 256 per rank, n 4096
        N=8, rs=dict(M=4096, k=256, n=4096, x=NORMAL1, w=NORMAL002, seed=3002),
        y_dtype="bf16", direction="uni", chunks=1),
    "gpt3_h12288_s2048_n8": dict(  # QKV AG-GEMM and attention-out GEMM-RS
        N=8, ag=dict(m=256, K=12288, n=4608, x=NORMAL1, w=NORMAL002, seed=4000),
        rs=dict(M=2048, k=1536, n=12288, x=NORMAL1, w=NORMAL002, seed=4002),
        y_dtype="bf16", direction="bidi", chunks=1),
    "mlp_h8192_ffn28672_s8192": dict(  # fc1 AG-GEMM and fc2 GEMM-RS; N, chunks, ring swept
        N=8, ag=dict(m=None, K=8192, n=None, x=NORMAL1, w=NORMAL002, seed=5000),
        rs=dict(M=8192, k=None, n=8192, x=NORMAL1, w=NORMAL002, seed=5002),
        y_dtype="bf16", direction="uni", chunks=1),
}

MLP_S, MLP_H, MLP_FFN = 8192, 8192, 28672


def mlp_shapes(N: int):
    """Per-rank shapes of the h=8192, ffn=28672, s=8192 MLP at N ranks."""
    assert MLP_S % N == 0 and MLP_FFN % N == 0
    return dict(ag=dict(m=MLP_S // N, K=MLP_H, n=MLP_FFN // N),
                rs=dict(M=MLP_S, k=MLP_FFN // N, n=MLP_H))
