"""The allocation-free AllGather->GEMM entry point, for callers that cannot
allocate device memory (a plugin handed only its inputs and outputs by a
framework that owns every allocation, or a loop where cudaMalloc is not
acceptable), against the regular entry point that takes a caller-allocated
workspace, and against the oracle.  Collected last on purpose, so that a run
stopping at the first failure has run every other test before it."""

import ctypes

import pytest
import torch

import oracle
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4   # the fp32-output bar of the parity tests
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _with_workspace(plan, xd, wd, N, m, K, n):
    ws = torch.full((plan.ag_workspace_size(m, K),), 0xFF, dtype=torch.uint8, device=DEV)
    y = torch.full((N, N * m, n), float("nan"), dtype=torch.float32, device=DEV)
    cm.cm_ag_gemm(plan, xd, wd, y, ws, "nk")
    st, info = cm.cm_check_status(ws)
    assert st == 0, (st, info)
    return y


def test_no_alloc_matches_workspace_entry_point_twice():
    """Two calls in a row share the library's scratch array.  The second one
    has other inputs and another shape, so it cannot pass on receive slots
    that still hold the first call's shards."""
    cases = [(4, 256, 512, 768, 2, 4242), (4, 320, 384, 512, 1, 4243)]
    for N, m, K, n, chunks, seed in cases:
        plan = cm.Plan(N, chunks, "uni")
        assert plan.ag_workspace_size(m, K) <= cm.CM_NOALLOC_SCRATCH_BYTES
        x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=seed, w_layout="nk")
        xd, wd = x.to(DEV), w.to(DEV)
        ref = _with_workspace(plan, xd, wd, N, m, K, n).double().cpu().numpy()
        exact = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
        y = torch.full((N, N * m, n), float("nan"), dtype=torch.float32, device=DEV)
        cm.cm_ag_gemm_noalloc(plan, xd, wd, y, "nk")
        st, info = cm.cm_ag_gemm_noalloc_check_status()
        assert st == 0, (st, info)
        yn = y.double().cpu().numpy()
        assert oracle.normwise_max_rel_err(yn, ref) <= TOL_F32
        assert oracle.normwise_max_rel_err(yn, exact) <= TOL_F32


def test_no_alloc_reports_a_device_timeout():
    """A rank that never forwards its shard: the consumers' bounded waits
    expire, the status accessor reports it, and the next call is correct."""
    N, m, K, n = 4, 128, 128, 256
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=17, w_layout="nk")
    xd, wd = x.to(DEV), w.to(DEV)
    plan = cm.Plan(N, 1, "uni")
    plan.set_option(cm.CM_OPT_TIMEOUT_NS, 50_000_000)
    plan.set_option(cm.CM_OPT_SKIP_SIGNAL, (cm.CM_OP_AG_GEMM << 16) | (1 << 8) | 0)
    y = torch.empty(N, N * m, n, dtype=torch.float32, device=DEV)
    cm.cm_ag_gemm_noalloc(plan, xd, wd, y, "nk")
    st, info = cm.cm_ag_gemm_noalloc_check_status()
    assert st == cm.CM_ERR_TIMEOUT and info[0] == cm.CM_ERR_TIMEOUT, (st, info)
    plan.set_option(cm.CM_OPT_SKIP_SIGNAL, -1)
    cm.cm_ag_gemm_noalloc(plan, xd, wd, y, "nk")
    st, info = cm.cm_ag_gemm_noalloc_check_status()
    assert st == 0, (st, info)
    exact = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    assert oracle.normwise_max_rel_err(y.double().cpu().numpy(), exact) <= TOL_F32


def test_no_alloc_rejects_problems_beyond_its_scratch():
    plan = cm.Plan(8, 1, "uni")
    m, K, n = 4096, 4096, 256        # 2*8*4096*4096*2 bytes of receive slots > 64 MiB
    assert plan.ag_workspace_size(m, K) > cm.CM_NOALLOC_SCRATCH_BYTES
    lib = cm.load()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = lib.cm_ag_gemm_noalloc(plan.handle, fake, fake, cm.CM_W_NK, fake, cm.CM_BF16, m, K, n, None)
    assert st == cm.CM_ERR_WORKSPACE
