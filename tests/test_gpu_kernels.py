"""Every tile kernel -- CTA pairs (tcgen05 cta_group::2, one pair per
cluster) and single CTAs -- against the oracle and against each other."""

import numpy as np
import pytest
import torch

import oracle
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen
from test_gpu_parity import TOL_F32, _np, run_ag, run_rs

pytestmark = pytest.mark.gpu

PAIR, SINGLE, PAIR_CL2 = 0, 1, 2
KERNELS = [PAIR, SINGLE, PAIR_CL2]


def _plan(N, chunks, direction, kernel):
    p = cm.Plan(N, chunks, direction)
    p.set_option(cm.CM_OPT_KERNEL, kernel)
    return p


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("N,m,K,n,chunks,direction", [
    (2, 64, 256, 512, 1, "uni"),        # rows per chunk below one CTA's 128
    (3, 200, 200, 296, 2, "bidi"),      # ragged rows / columns / K
    (4, 384, 320, 768, 1, "uni"),       # row tiles straddling the pair split; 3 column tiles
    (5, 136, 72, 520, 1, "none"),       # odd column-tile count
    (2, 48, 64, 256, 1, "uni"),         # rows below half a CTA's 128, one column tile
])
@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_kernel_vs_oracle(kernel, N, m, K, n, chunks, direction, layout):
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=m + K, w_layout=layout)
    ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), layout)
    y, _, _ = run_ag(_plan(N, chunks, direction, kernel), x, w, layout)
    assert oracle.normwise_max_rel_err(_np(y), ref) <= TOL_F32
    xr, wr = gen.rs_inputs(N, N * m, K, n, gen.NORMAL1, gen.NORMAL002, seed=m + K + 1, w_layout=layout)
    refr = oracle.gemm_rs(gen.bf16_bits(xr), gen.bf16_bits(wr), layout)
    yr, _, _ = run_rs(_plan(N, chunks, direction, kernel), xr, wr, layout)
    assert oracle.normwise_max_rel_err(_np(yr), refr) <= TOL_F32


def test_kernels_agree_bitwise_on_ag():
    N, m, K, n = 4, 512, 1024, 1280
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=99, w_layout="nk")
    base, _, _ = run_ag(_plan(N, 1, "uni", SINGLE), x, w, "nk")
    for k in (PAIR, PAIR_CL2):
        y, _, _ = run_ag(_plan(N, 1, "uni", k), x, w, "nk")
        assert torch.equal(y, base), k


@pytest.mark.parametrize("hints,promotion", [(0x01, 3), (0x21, 0), (0x12, 2)])
def test_l2_options_change_no_bits(hints, promotion):
    """Cache-priority hints and L2 promotion only steer caching: same bits out."""
    N, m, K, n = 4, 320, 512, 768
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=7, w_layout="nk")
    xr, wr = gen.rs_inputs(N, N * m, K, n, gen.NORMAL1, gen.NORMAL002, seed=8, w_layout="kn")
    base, _, _ = run_ag(_plan(N, 1, "uni", PAIR), x, w, "nk")
    base_r, _, _ = run_rs(_plan(N, 1, "uni", PAIR), xr, wr, "kn")
    p = _plan(N, 1, "uni", PAIR)
    p.set_option(cm.CM_OPT_L2_HINTS, hints)
    p.set_option(cm.CM_OPT_L2_PROMOTION, promotion)
    y, _, _ = run_ag(p, x, w, "nk")
    yr, _, _ = run_rs(p, xr, wr, "kn")
    assert torch.equal(y, base)
    assert torch.equal(yr, base_r)


@pytest.mark.parametrize("kernel", [PAIR, SINGLE])
@pytest.mark.parametrize("band", [1, 3])
def test_row_bands_change_no_bits(kernel, band):
    """The row-band tile order only reorders tiles: same bits out."""
    N, m, K, n = 4, 320, 256, 1280
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=17, w_layout="nk")
    xr, wr = gen.rs_inputs(N, N * m, K, n, gen.NORMAL1, gen.NORMAL002, seed=18, w_layout="nk")
    base, _, _ = run_ag(_plan(N, 2, "uni", kernel), x, w, "nk")
    base_r, _, _ = run_rs(_plan(N, 2, "uni", kernel), xr, wr, "nk")
    p = _plan(N, 2, "uni", kernel)
    p.set_option(cm.CM_OPT_ROW_BAND, band)
    y, _, _ = run_ag(p, x, w, "nk")
    yr, _, _ = run_rs(p, xr, wr, "nk")
    assert torch.equal(y, base)
    assert torch.equal(yr, base_r)
    ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    assert oracle.normwise_max_rel_err(_np(y), ref) <= TOL_F32


@pytest.mark.parametrize("kernel", KERNELS)
def test_tagged_placement_each_kernel(kernel):
    N, m, K, n = 8, 384, 64, 512
    x, w = gen.tagged_ag_inputs(N, m, K, n, "nk")
    ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    for direction, chunks in (("uni", 1), ("bidi", 2), ("uni", 4)):
        y, _, _ = run_ag(_plan(N, chunks, direction, kernel), x, w, "nk", torch.bfloat16)
        assert np.array_equal(_np(y), ref)


@pytest.mark.parametrize("kernel", KERNELS)
def test_timeout_each_kernel(kernel):
    N = 4
    x, w = gen.ag_inputs(N, 256, 128, 256, gen.NORMAL1, gen.NORMAL002, seed=3, w_layout="nk")
    p = _plan(N, 1, "uni", kernel)
    p.set_option(cm.CM_OPT_TIMEOUT_NS, 50_000_000)
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, (cm.CM_OP_AG_GEMM << 16) | (1 << 8) | 0)
    _, st, info = run_ag(p, x, w, "nk", check=False)
    assert st == cm.CM_ERR_TIMEOUT, (st, info)
    xr, wr = gen.rs_inputs(N, 1024, 128, 256, gen.NORMAL1, gen.NORMAL002, seed=4, w_layout="nk")
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, (cm.CM_OP_GEMM_RS << 16) | (2 << 8) | 1)
    _, st, info = run_rs(p, xr, wr, "nk", check=False)
    assert st == cm.CM_ERR_TIMEOUT, (st, info)
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, -1)
    ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    y, _, _ = run_ag(p, x, w, "nk")
    assert oracle.normwise_max_rel_err(_np(y), ref) <= TOL_F32

