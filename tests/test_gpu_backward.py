"""GPU parity of the backward pair of the column-parallel layer ("Tensor
Parallelism > Communication Patterns": the backward is the forward's dual;
"Hiding Tensor-Parallel Collectives: AG/RS Overlap in Megatron", section 7:
bulk overlap) against the fp64 oracle:

* data gradient   dX = the GEMM->ReduceScatter of dY_r @ W_r (W_r read [n][K]);
* weight gradient dW_r = dY_r^T @ concat_j(X_j), after an AllGather that runs
  on a second stream under the data-gradient GEMM-RS.

Bars: normwise max relative error <= 2e-2 (bf16 out), <= 1e-4 (fp32 out);
exact on small-integer inputs; bulk overlap on or off gives the same bits."""

import numpy as np
import pytest
import torch

import oracle
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen
from test_gpu_parity import DEV, TOL, TOL_F32, _np

pytestmark = pytest.mark.gpu


def backward_inputs(N, m, K, n, seed):
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=seed, w_layout="nk")   # w [N][n][K]
    dy, _ = gen.ag_inputs(N, N * m, n, 1, gen.NORMAL1, gen.NORMAL1, seed=seed + 1)           # [N][N*m][n]
    return x, w, dy


def run_backward(plan, x, w, dy, dtype=torch.float32, stream=None, overlap=1):
    N, m, K = x.shape
    n = w.shape[1]
    plan.set_option(cm.CM_OPT_BULK_OVERLAP, overlap)
    ws = torch.full((plan.backward_pair_workspace_size(m, K, n),), 0xFF, dtype=torch.uint8, device=DEV)
    dx = torch.full((N, m, K), float("nan"), dtype=dtype, device=DEV)
    dw = torch.full((N, n, K), float("nan"), dtype=dtype, device=DEV)
    cm.cm_backward_pair(plan, x.to(DEV), w.to(DEV), dy.to(DEV), dx, dw, ws, stream)
    st, info = cm.cm_check_status(ws, stream)
    assert st == 0, f"status {st} info {info}"
    return dx, dw


def oracle_backward(x, w, dy):
    xb, wb, dyb = gen.bf16_bits(x), gen.bf16_bits(w), gen.bf16_bits(dy)
    return oracle.gemm_rs(dyb, wb, "kn"), oracle.wgrad(xb, dyb)


@pytest.mark.parametrize("N,m,K,n,chunks,direction", [
    (1, 128, 256, 256, 1, "uni"),       # one rank: both gradients are plain GEMMs
    (2, 64, 256, 512, 1, "uni"),
    (2, 48, 136, 200, 1, "uni"),        # ragged K and n; 96 tokens
    (3, 96, 320, 264, 2, "bidi"),
    (4, 256, 512, 768, 2, "uni"),
    (8, 128, 256, 384, 1, "bidi"),
])
def test_backward_pair_vs_oracle(N, m, K, n, chunks, direction):
    x, w, dy = backward_inputs(N, m, K, n, seed=N * 1000 + m)
    ref_dx, ref_dw = oracle_backward(x, w, dy)
    dx, dw = run_backward(cm.Plan(N, chunks, direction), x, w, dy)
    assert oracle.normwise_max_rel_err(_np(dx), ref_dx) <= TOL_F32
    assert oracle.normwise_max_rel_err(_np(dw), ref_dw) <= TOL_F32
    dxb, dwb = run_backward(cm.Plan(N, chunks, direction), x, w, dy, torch.bfloat16)
    assert oracle.normwise_max_rel_err(_np(dxb), ref_dx) <= TOL
    assert oracle.normwise_max_rel_err(_np(dwb), ref_dw) <= TOL


@pytest.mark.parametrize("N", [1, 2, 4])
def test_backward_pair_exact_on_integers(N):
    m, K, n = 64, 192, 128
    g = torch.Generator().manual_seed(N)
    x = torch.randint(-3, 4, (N, m, K), generator=g).to(torch.bfloat16)
    w = torch.randint(-3, 4, (N, n, K), generator=g).to(torch.bfloat16)
    dy = torch.randint(-3, 4, (N, N * m, n), generator=g).to(torch.bfloat16)
    ref_dx, ref_dw = oracle_backward(x, w, dy)
    dx, dw = run_backward(cm.Plan(N, 1, "uni"), x, w, dy)
    assert np.array_equal(_np(dx), ref_dx)
    assert np.array_equal(_np(dw), ref_dw)


def test_bulk_overlap_changes_no_bits():
    N, m, K, n = 4, 256, 512, 512
    x, w, dy = backward_inputs(N, m, K, n, seed=5)
    a = run_backward(cm.Plan(N, 1, "uni"), x, w, dy, overlap=1)
    b = run_backward(cm.Plan(N, 1, "uni"), x, w, dy, overlap=0)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_back_to_back_on_a_user_stream():
    """Two calls queued on one stream share a workspace; the second call's
    gather must not overwrite what the first call's weight gradient reads."""
    N, m, K, n = 4, 128, 256, 384
    sets = [backward_inputs(N, m, K, n, seed=s) for s in (11, 12)]
    refs = [oracle_backward(*t) for t in sets]
    plan = cm.Plan(N, 1, "uni")
    ws = torch.full((plan.backward_pair_workspace_size(m, K, n),), 0xFF, dtype=torch.uint8, device=DEV)
    outs = [(torch.empty(N, m, K, device=DEV), torch.empty(N, n, K, device=DEV)) for _ in sets]
    dev_in = [tuple(t.to(DEV) for t in s_) for s_ in sets]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for (x, w, dy), (dx, dw) in zip(dev_in, outs):
            cm.cm_backward_pair(plan, x, w, dy, dx, dw, ws, s)
        snap = [(dx.clone(), dw.clone()) for dx, dw in outs]
    st, _ = cm.cm_check_status(ws, s)
    assert st == 0
    for (dx, dw), (rdx, rdw) in zip(snap, refs):
        assert oracle.normwise_max_rel_err(_np(dx), rdx) <= TOL_F32
        assert oracle.normwise_max_rel_err(_np(dw), rdw) <= TOL_F32


def test_shape_errors():
    plan = cm.Plan(2, 1, "uni")
    x = torch.zeros(2, 16, 64, dtype=torch.bfloat16, device=DEV)     # 32 tokens < 64
    w = torch.zeros(2, 64, 64, dtype=torch.bfloat16, device=DEV)
    dy = torch.zeros(2, 32, 64, dtype=torch.bfloat16, device=DEV)
    ws = torch.full((plan.backward_pair_workspace_size(16, 64, 64),), 0xFF, dtype=torch.uint8, device=DEV)
    dx, dw = torch.empty(2, 16, 64, device=DEV), torch.empty(2, 64, 64, device=DEV)
    with pytest.raises(cm.CMError):
        cm.cm_backward_pair(plan, x, w, dy, dx, dw, ws)


def test_full_size_sampled_rows():
    """The backward of the MLP fc1 (h=8192, ffn=28672, s=8192) at N=8."""
    N = 8
    sh = gen.mlp_shapes(N)["ag"]
    m, K, n = sh["m"], sh["K"], sh["n"]
    x, w, dy = backward_inputs(N, m, K, n, seed=6000)
    dx, dw = run_backward(cm.Plan(N, 1, "uni"), x, w, dy, torch.bfloat16)
    rng = np.random.default_rng(2)
    xb, wb, dyb = gen.bf16_bits(x), gen.bf16_bits(w), gen.bf16_bits(dy)
    owners = np.concatenate([np.arange(N), rng.integers(0, N, 8)])
    rows = np.concatenate([np.full(N, m - 1), rng.integers(0, m, 8)])
    ref = oracle.gemm_rs_rows(dyb, wb, owners, rows, "kn")
    got = dx[torch.as_tensor(owners, device=DEV), torch.as_tensor(rows, device=DEV)]
    assert oracle.normwise_max_rel_err(_np(got), ref) <= TOL
    ranks = np.concatenate([np.arange(N), rng.integers(0, N, 4)])
    wrows = np.concatenate([np.full(N, n - 1), rng.integers(0, n, 4)])
    ref = oracle.wgrad_rows(xb, dyb, ranks, wrows)
    got = dw[torch.as_tensor(ranks, device=DEV), torch.as_tensor(wrows, device=DEV)]
    assert oracle.normwise_max_rel_err(_np(got), ref) <= TOL
    assert torch.isfinite(dx).all() and torch.isfinite(dw).all()
