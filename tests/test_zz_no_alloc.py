"""The allocation-free AllGather->GEMM entry point, for callers that cannot
allocate device memory, against the regular entry point that takes a
caller-allocated workspace.  Collected last on purpose."""

import ctypes

import pytest
import torch

import oracle
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4   # the fp32-output bar of the parity tests


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def test_no_alloc_matches_workspace_entry_point_twice():
    dev = "cuda:0"
    N, m, K, n = 4, 256, 512, 768
    plan = cm.Plan(N, 2, "uni")
    assert plan.ag_workspace_size(m, K) <= cm.CM_NOALLOC_SCRATCH_BYTES
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=4242, w_layout="nk")
    xd, wd = x.to(dev), w.to(dev)
    ws = torch.empty(plan.ag_workspace_size(m, K), dtype=torch.uint8, device=dev)
    ref = torch.empty(N, N * m, n, dtype=torch.float32, device=dev)
    cm.cm_ag_gemm(plan, xd, wd, ref, ws, "nk")
    st, info = cm.cm_check_status(ws)
    assert st == 0, (st, info)
    exact = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    for _ in range(2):   # two calls in a row share the library's scratch array
        y = torch.full((N, N * m, n), float("nan"), dtype=torch.float32, device=dev)
        cm.cm_ag_gemm_noalloc(plan, xd, wd, y, "nk")
        torch.cuda.synchronize()
        yn = y.double().cpu().numpy()
        assert oracle.normwise_max_rel_err(yn, ref.double().cpu().numpy()) <= TOL_F32
        assert oracle.normwise_max_rel_err(yn, exact) <= TOL_F32


def test_no_alloc_rejects_problems_beyond_its_scratch():
    plan = cm.Plan(8, 1, "uni")
    m, K, n = 4096, 4096, 256        # 2*8*4096*4096*2 bytes of receive slots > 64 MiB
    assert plan.ag_workspace_size(m, K) > cm.CM_NOALLOC_SCRATCH_BYTES
    lib = cm.load()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = lib.cm_ag_gemm_noalloc(plan.handle, fake, fake, cm.CM_W_NK, fake, cm.CM_BF16, m, K, n, None)
    assert st == cm.CM_ERR_WORKSPACE
