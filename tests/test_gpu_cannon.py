"""GPU parity of Cannon-style 2-D rotation ("Overlap Communication with
Dependent Computation via Decomposition in Large Deep Learning Models",
section "What people did before") against the fp64 oracle: the plain GEMM of
the assembled blocks, and the rank-by-rank rotation simulation.

Bars: normwise max relative error <= 1e-4 (fp32 out) and <= 2e-2 (bf16 out);
exact on small-integer inputs (every block product and the fp32 sum over
steps are exact integers)."""

import numpy as np
import pytest
import torch

import oracle
from oracle import ring
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen
from test_gpu_parity import DEV, TOL, TOL_F32, _np

pytestmark = pytest.mark.gpu


def blocks(q, bm, bk, bn, seed, layout="nk"):
    a, _ = gen.ag_inputs(q * q, bm, bk, 1, gen.NORMAL1, gen.NORMAL002, seed=seed)
    shape = (q * q, bn, bk) if layout == "nk" else (q * q, bk, bn)
    b, _ = gen.ag_inputs(shape[0], shape[1], shape[2], 1, gen.NORMAL1, gen.NORMAL002, seed=seed + 1)
    return a, b


def assembled_ref(a, b, q, layout):
    """C = A @ B of the assembled matrices, returned as blocks [q*q][bm][bn]."""
    P, bm, bk = a.shape
    A = a.reshape(q, q, bm, bk).permute(0, 2, 1, 3).reshape(q * bm, q * bk).contiguous()
    bb = b if layout == "kn" else b.transpose(1, 2)
    bn = bb.shape[2]
    B = bb.reshape(q, q, bk, bn).permute(0, 2, 1, 3).reshape(q * bk, q * bn).contiguous()
    C = oracle.gemm(gen.bf16_bits(A), gen.bf16_bits(B), "kn")
    return C.reshape(q, bm, q, bn).transpose(0, 2, 1, 3).reshape(P, bm, bn)


def run_cannon(plan, a, b, layout="nk", dtype=torch.float32, stream=None):
    P, bm, bk = a.shape
    bn = b.shape[1] if layout == "nk" else b.shape[2]
    ws = torch.full((plan.cannon_workspace_size(bm, bk, bn),), 0xFF, dtype=torch.uint8, device=DEV)
    c = torch.full((P, bm, bn), float("nan"), dtype=dtype, device=DEV)
    cm.cm_cannon_gemm(plan, a.to(DEV), b.to(DEV), c, ws, layout, stream)
    st, info = cm.cm_check_status(ws, stream)
    assert st == 0, f"status {st} info {info}"
    return c


@pytest.mark.parametrize("q,bm,bk,bn", [
    (1, 256, 256, 512),
    (2, 128, 256, 256),
    (2, 200, 136, 296),       # ragged rows, K and columns
    (3, 96, 192, 264),
    (4, 256, 512, 512),
])
@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_cannon_vs_oracle(q, bm, bk, bn, layout):
    a, b = blocks(q, bm, bk, bn, seed=q * 100 + bm, layout=layout)
    ref = assembled_ref(a, b, q, layout)
    c = run_cannon(cm.Plan(q * q, 1, "uni"), a, b, layout)
    assert oracle.normwise_max_rel_err(_np(c), ref) <= TOL_F32
    cb = run_cannon(cm.Plan(q * q, 1, "uni"), a, b, layout, torch.bfloat16)
    assert oracle.normwise_max_rel_err(_np(cb), ref) <= TOL


def test_cannon_matches_rotation_simulation():
    q, bm, bk, bn = 3, 64, 128, 128
    a, b = blocks(q, bm, bk, bn, seed=7)
    sim = ring.cannon_gemm(gen.bf16_bits(a), gen.bf16_bits(b), q, "nk")
    c = run_cannon(cm.Plan(q * q, 1, "uni"), a, b)
    assert oracle.normwise_max_rel_err(_np(c), sim) <= TOL_F32


@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("q", [2, 4])
def test_cannon_exact_on_integers(kernel, q):
    bm, bk, bn = 128, 64, 256
    g = torch.Generator().manual_seed(q)
    a = torch.randint(-3, 4, (q * q, bm, bk), generator=g).to(torch.bfloat16)
    b = torch.randint(-3, 4, (q * q, bn, bk), generator=g).to(torch.bfloat16)
    ref = assembled_ref(a, b, q, "nk")
    p = cm.Plan(q * q, 1, "uni")
    p.set_option(cm.CM_OPT_KERNEL, kernel)
    c = run_cannon(p, a, b)
    assert np.array_equal(_np(c), ref)


def test_cannon_back_to_back_on_a_user_stream():
    q, bm, bk, bn = 2, 128, 256, 256
    sets = [blocks(q, bm, bk, bn, seed=s) for s in (21, 22)]
    refs = [assembled_ref(a, b, q, "nk") for a, b in sets]
    plan = cm.Plan(q * q, 1, "uni")
    ws = torch.full((plan.cannon_workspace_size(bm, bk, bn),), 0xFF, dtype=torch.uint8, device=DEV)
    outs = [torch.empty(q * q, bm, bn, device=DEV) for _ in sets]
    dev_in = [(a.to(DEV), b.to(DEV)) for a, b in sets]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for (a, b), c in zip(dev_in, outs):
            cm.cm_cannon_gemm(plan, a, b, c, ws, "nk", s)
        snap = [c.clone() for c in outs]
    st, _ = cm.cm_check_status(ws, s)
    assert st == 0
    for got, ref in zip(snap, refs):
        assert oracle.normwise_max_rel_err(_np(got), ref) <= TOL_F32


def test_cannon_needs_a_square_grid():
    plan = cm.Plan(8, 1, "uni")
    assert plan.cannon_workspace_size(64, 64, 64) == 0
    a = torch.zeros(8, 64, 64, dtype=torch.bfloat16, device=DEV)
    c = torch.zeros(8, 64, 64, device=DEV)
    ws = torch.full((1 << 20,), 0xFF, dtype=torch.uint8, device=DEV)
    with pytest.raises(cm.CMError):
        cm.cm_cannon_gemm(plan, a, a, c, ws)
