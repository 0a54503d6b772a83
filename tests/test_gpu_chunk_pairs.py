"""Chunks of at most 128 rows on the CTA-pair kernel: two consecutive chunks
share one 256-row pair tile, one per CTA, each CTA with its own chunk's
readiness flags.  Against the oracle (AllGather->GEMM and
GEMM->ReduceScatter, both rings, both weight layouts, odd chunk counts that
cannot pair), bit-exact on tagged and integer inputs, bit-identical to the
one-chunk AllGather, and with a dropped signal that must time out."""

import numpy as np
import pytest
import torch

import oracle
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen
from test_gpu_parity import TOL_F32, _np, run_ag, run_rs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,m,K,n,chunks,direction", [
    (4, 256, 320, 768, 2, "uni"),      # 128-row chunks: the pair covers chunks 2g, 2g+1
    (4, 256, 320, 768, 4, "bidi"),     # 64-row chunks
    (3, 360, 200, 296, 4, "uni"),      # 90-row chunks, ragged K and columns
    (5, 240, 136, 520, 8, "bidi"),     # 30-row chunks, odd rank count
    (2, 384, 256, 512, 3, "uni"),      # odd chunk count: no pairing
    (6, 200, 128, 256, 2, "uni"),      # 100-row chunks
])
@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_small_chunks_vs_oracle(N, m, K, n, chunks, direction, layout):
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=m + chunks, w_layout=layout)
    ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), layout)
    y, _, _ = run_ag(cm.Plan(N, chunks, direction), x, w, layout)
    assert oracle.normwise_max_rel_err(_np(y), ref) <= TOL_F32
    xr, wr = gen.rs_inputs(N, N * m, K, n, gen.NORMAL1, gen.NORMAL002, seed=m + chunks + 1, w_layout=layout)
    refr = oracle.gemm_rs(gen.bf16_bits(xr), gen.bf16_bits(wr), layout)
    yr, _, _ = run_rs(cm.Plan(N, chunks, direction), xr, wr, layout)
    assert oracle.normwise_max_rel_err(_np(yr), refr) <= TOL_F32


@pytest.mark.parametrize("chunks", [2, 4, 8])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
def test_small_chunks_placement_and_ag_bits(chunks, direction):
    """Tagged inputs place every shard row exactly; and the AllGather result
    is bit-identical to the one-chunk schedule."""
    N, m, K, n = 4, 256, 64, 512
    x, w = gen.tagged_ag_inputs(N, m, K, n, "nk")
    ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    y, _, _ = run_ag(cm.Plan(N, chunks, direction), x, w, "nk")
    assert np.array_equal(_np(y), ref)
    xs, ws = gen.ag_inputs(N, m, 512, n, gen.NORMAL1, gen.NORMAL002, seed=chunks, w_layout="nk")
    base, _, _ = run_ag(cm.Plan(N, 1, direction), xs, ws, "nk")
    yc, _, _ = run_ag(cm.Plan(N, chunks, direction), xs, ws, "nk")
    assert torch.equal(yc, base)


@pytest.mark.parametrize("chunks,direction", [(2, "uni"), (4, "bidi")])
def test_small_chunks_rs_exact_on_integers(chunks, direction):
    N, M, k, n = 4, 1024, 128, 512
    g = torch.Generator().manual_seed(chunks)
    x = torch.randint(-3, 4, (N, M, k), generator=g).to(torch.bfloat16)
    w = torch.randint(-2, 3, (N, n, k), generator=g).to(torch.bfloat16)
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    y, _, _ = run_rs(cm.Plan(N, chunks, direction), x, w, "nk")
    assert np.array_equal(_np(y), ref)


def test_small_chunks_serial_steps_and_few_ctas():
    """Step-serial launches and a 7-CTA grid (many tiles per pair) give the
    same AllGather bits."""
    N, m, K, n = 4, 256, 256, 768
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=5, w_layout="nk")
    base, _, _ = run_ag(cm.Plan(N, 1, "uni"), x, w, "nk")
    p = cm.Plan(N, 4, "uni")
    p.set_option(cm.CM_OPT_SERIAL_STEPS, 1)
    y, _, _ = run_ag(p, x, w, "nk")
    assert torch.equal(y, base)
    p = cm.Plan(N, 4, "bidi")
    p.set_option(cm.CM_OPT_GRID, 8)
    y, _, _ = run_ag(p, x, w, "nk")
    assert torch.equal(y, base)


@pytest.mark.parametrize("op", ["ag", "rs"])
def test_small_chunks_skipped_signal_times_out(op):
    N, m, K, n = 4, 256, 128, 512
    p = cm.Plan(N, 4, "uni")
    p.set_option(cm.CM_OPT_TIMEOUT_NS, 50_000_000)
    code = cm.CM_OP_AG_GEMM if op == "ag" else cm.CM_OP_GEMM_RS
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, (code << 16) | (1 << 8) | 0)
    if op == "ag":
        x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=9, w_layout="nk")
        _, st, info = run_ag(p, x, w, "nk", check=False)
    else:
        x, w = gen.rs_inputs(N, N * m, K, n, gen.NORMAL1, gen.NORMAL002, seed=9, w_layout="nk")
        _, st, info = run_rs(p, x, w, "nk", check=False)
    assert st == cm.CM_ERR_TIMEOUT, (st, info)
