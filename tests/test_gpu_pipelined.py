"""GPU parity of the pipelined GEMM->ReduceScatter ("Hiding Tensor-Parallel
Collectives: AG/RS Overlap in Megatron", section 6: the GEMM in chunks, the
ReduceScatter of chunk j under the GEMM of chunk j+1) against the fp64
oracle's GEMM->ReduceScatter definition, and against the moving-bucket RS.

Bars as for the moving-bucket RS: normwise max relative error <= 2e-2
(bf16 out) and <= 1e-4 (fp32 out); exact on small-integer inputs, where every
fp32 partial and every sum over ranks is an exactly representable integer."""

import numpy as np
import pytest
import torch

import oracle
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen
from test_gpu_parity import DEV, TOL, TOL_F32, _np, run_rs

pytestmark = pytest.mark.gpu

PAIR, SINGLE = 0, 1


def run_pipe(plan, x, w, layout="nk", ydtype=torch.float32, stream=None):
    N, M, k = x.shape
    n = w.shape[1] if layout == "nk" else w.shape[2]
    ws = torch.full((plan.rs_pipelined_workspace_size(M, n),), 0xFF, dtype=torch.uint8, device=DEV)
    y = torch.full((N, M // N, n), float("nan"), dtype=ydtype, device=DEV)
    cm.cm_gemm_rs_pipelined(plan, x.to(DEV), w.to(DEV), y, ws, layout, stream)
    st, info = cm.cm_check_status(ws, stream)
    assert st == 0, f"status {st} info {info}"
    return y


@pytest.mark.parametrize("N,M,k,n,chunks", [
    (1, 256, 128, 512, 1),        # one rank: a plain GEMM in one chunk
    (2, 128, 128, 512, 1),
    (2, 512, 200, 296, 2),        # ragged k and n
    (3, 768, 136, 520, 4),        # odd N; chunks of 64 rows; odd column-tile count
    (4, 2048, 320, 768, 2),       # several row tiles per chunk
    (8, 4096, 256, 1024, 4),
])
@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_pipelined_vs_oracle(N, M, k, n, chunks, layout):
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=M + k + n, w_layout=layout)
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), layout)
    y = run_pipe(cm.Plan(N, chunks, "uni"), x, w, layout)
    assert oracle.normwise_max_rel_err(_np(y), ref) <= TOL_F32
    yb = run_pipe(cm.Plan(N, chunks, "uni"), x, w, layout, torch.bfloat16)
    assert oracle.normwise_max_rel_err(_np(yb), ref) <= TOL


@pytest.mark.parametrize("kernel", [PAIR, SINGLE])
@pytest.mark.parametrize("chunks", [1, 2, 4])
def test_pipelined_exact_on_integers(kernel, chunks):
    """Small integers: products and sums are exact in fp32, so the output is
    the oracle's exactly, whatever the chunking and summation order."""
    N, M, k, n = 4, 1024, 96, 640
    x = torch.randint(-3, 4, (N, M, k), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    w = torch.randint(-3, 4, (N, n, k), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    p = cm.Plan(N, chunks, "uni")
    p.set_option(cm.CM_OPT_KERNEL, kernel)
    y = run_pipe(p, x, w, "nk")
    assert np.array_equal(_np(y), ref)


def test_pipelined_matches_moving_bucket():
    N, M, k, n = 8, 2048, 512, 1536
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=77, w_layout="nk")
    y_ring, _, _ = run_rs(cm.Plan(N, 2, "uni"), x, w, "nk")
    y_pipe = run_pipe(cm.Plan(N, 2, "uni"), x, w, "nk")
    # same products, fp32 sums in a different order
    assert oracle.normwise_max_rel_err(_np(y_pipe), _np(y_ring)) <= TOL_F32


def test_back_to_back_calls_on_a_side_stream():
    """Two calls queued on a user stream share one workspace: the second GEMM
    must not overwrite partials the first call's last reduction still reads."""
    N, M, k, n = 4, 2048, 256, 1024
    s = torch.cuda.Stream()
    xs = [gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=s_, w_layout="nk") for s_ in (5, 6)]
    refs = [oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk") for x, w in xs]
    plan = cm.Plan(N, 4, "uni")
    ws = torch.full((plan.rs_pipelined_workspace_size(M, n),), 0xFF, dtype=torch.uint8, device=DEV)
    ys = [torch.full((N, M // N, n), float("nan"), device=DEV) for _ in xs]
    dev_in = [(x.to(DEV), w.to(DEV)) for x, w in xs]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for (x, w), y in zip(dev_in, ys):
            cm.cm_gemm_rs_pipelined(plan, x, w, y, ws, "nk", s)
        snap = [y.clone() for y in ys]   # queued on s: sees the results only if the reductions are ordered
    st, _ = cm.cm_check_status(ws, s)
    assert st == 0
    for got, ref in zip(snap, refs):
        assert oracle.normwise_max_rel_err(_np(got), ref) <= TOL_F32


def test_full_size_sampled_rows():
    """The MLP h=8192, ffn=28672, s=8192 fc2 at N=8 with 4 pipeline chunks."""
    N = 8
    sh = gen.mlp_shapes(N)["rs"]
    M, k, n = sh["M"], sh["k"], sh["n"]
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=5002, w_layout="nk")
    y = run_pipe(cm.Plan(N, 4, "uni"), x, w, "nk", torch.bfloat16)
    rng = np.random.default_rng(1)
    Mb = M // N
    owners = np.concatenate([np.arange(N), np.arange(N), rng.integers(0, N, 16)])
    rows = np.concatenate([np.zeros(N, int), np.full(N, Mb - 1), rng.integers(0, Mb, 16)])
    ref = oracle.gemm_rs_rows(gen.bf16_bits(x), gen.bf16_bits(w), owners, rows, "nk")
    got = y[torch.as_tensor(owners, device=DEV), torch.as_tensor(rows, device=DEV)]
    assert oracle.normwise_max_rel_err(_np(got), ref) <= TOL
    assert torch.isfinite(y).all()
