"""The bounds-checked build of the library (CM_DEBUG_BOUNDS): every computed
flag, slot, row and buffer index is compared in the kernels with the extent
of its buffer, and one outside it is reported as CM_ERR_BOUNDS (with the
task, chunk and which index) instead of being used.

* It reports nothing on correct calls and gives the release build's bits
  (the checks change no arithmetic), on every entry point and kernel.
* A planted mistake -- done signals moved beyond the flag words by
  CM_OPT_DEBUG_FLAG_OFFSET, an option only this build accepts -- is turned
  into CM_ERR_BOUNDS, and the next call is correct.  The planted signals
  would otherwise land inside the same workspace (its bucket buffers follow
  the flag words and are far larger), so even an unchecked run would write
  only memory the call owns."""

import pytest
import torch

import oracle
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen
from test_gpu_parity import DEV, TOL_F32, _np

pytestmark = pytest.mark.gpu

KSITE_BOUNDS_FLAG = 16


@pytest.fixture(scope="module")
def dbg():
    import __graft_entry__
    __graft_entry__.build()
    return cm.bounds_checked()


def _ws(size):
    return torch.full((size,), 0xFF, dtype=torch.uint8, device=DEV)


def _ag(mod, plan, x, w, ydtype=torch.float32):
    N, m, K = x.shape
    n = w.shape[1]
    ws = _ws(plan.ag_workspace_size(m, K))
    y = torch.full((N, N * m, n), float("nan"), dtype=ydtype, device=DEV)
    mod.cm_ag_gemm(plan, x.to(DEV), w.to(DEV), y, ws, "nk")
    return y, mod.cm_check_status(ws)


def _rs(mod, plan, x, w, ydtype=torch.float32):
    N, M, k = x.shape
    n = w.shape[1]
    ws = _ws(plan.rs_workspace_size(M, n))
    y = torch.full((N, M // N, n), float("nan"), dtype=ydtype, device=DEV)
    mod.cm_gemm_rs(plan, x.to(DEV), w.to(DEV), y, ws, "nk")
    return y, mod.cm_check_status(ws)


def _plan(mod, N, chunks, direction, **opts):
    p = mod.Plan(N, chunks, direction)
    for k, v in opts.items():
        p.set_option(getattr(mod, k), v)
    return p


def test_version_names_the_bounds_checks(dbg):
    assert "bounds-checked" in dbg.version()
    assert "bounds-checked" not in cm.version()


@pytest.mark.parametrize("N,chunks,direction,opts", [
    (4, 1, "uni", {}),
    (4, 4, "uni", {}),                                  # 64-row chunks: two per pair tile
    (5, 2, "bidi", {}),
    (4, 2, "uni", {"CM_OPT_KERNEL": 1}),                # single-CTA kernel
    (8, 1, "uni", {"CM_OPT_TASK_ORDER": 2}),
])
def test_ag_same_bits_no_report(dbg, N, chunks, direction, opts):
    m, K, n = 256, 320, 520
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=N + chunks, w_layout="nk")
    yd, (st, info) = _ag(dbg, _plan(dbg, N, chunks, direction, **opts), x, w)
    assert st == 0, (st, info)
    yr, (st, info) = _ag(cm, _plan(cm, N, chunks, direction, **opts), x, w)
    assert st == 0, (st, info)
    assert torch.equal(yd, yr)


@pytest.mark.parametrize("N,chunks,direction,opts", [
    (4, 1, "uni", {"CM_OPT_RS_EPILOGUE": 1}),
    (4, 2, "uni", {"CM_OPT_RS_EPILOGUE": 2}),
    (8, 4, "uni", {"CM_OPT_RS_EPILOGUE": 2}),           # chunk pairs, two warp groups
    (8, 4, "uni", {"CM_OPT_RS_EPILOGUE": 3}),           # chunk pairs, every warp with vector adds
    (5, 1, "bidi", {"CM_OPT_RS_BUCKET_HINT": 2}),       # TMA epilogue with an L2 policy
    (4, 2, "bidi", {"CM_OPT_RS_EPILOGUE": 3, "CM_OPT_RS_IN_PLACE": 0}),
    (5, 1, "bidi", {"CM_OPT_RS_EPILOGUE": 1, "CM_OPT_RS_PRELOAD": 1}),
    (4, 2, "bidi", {"CM_OPT_RS_IN_PLACE": 0, "CM_OPT_RS_PRELOAD": 3}),
    (4, 1, "uni", {"CM_OPT_KERNEL": 1}),
])
def test_rs_same_bits_no_report(dbg, N, chunks, direction, opts):
    M, k, n = N * 256, 192, 776
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=N + 3 * chunks, w_layout="nk")
    yd, (st, info) = _rs(dbg, _plan(dbg, N, chunks, direction, **opts), x, w)
    assert st == 0, (st, info)
    yr, (st, info) = _rs(cm, _plan(cm, N, chunks, direction, **opts), x, w)
    assert st == 0, (st, info)
    assert torch.equal(yd, yr)


def test_other_entry_points_no_report(dbg):
    """Pipelined GEMM-RS, the backward pair and Cannon under the checks."""
    N, M, k, n = 4, 1024, 128, 512
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=41, w_layout="nk")
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    p = dbg.Plan(N, 4, "uni")
    ws = _ws(p.rs_pipelined_workspace_size(M, n))
    y = torch.empty(N, M // N, n, device=DEV)
    dbg.cm_gemm_rs_pipelined(p, x.to(DEV), w.to(DEV), y, ws, "nk")
    st, info = dbg.cm_check_status(ws)
    assert st == 0, (st, info)
    assert oracle.normwise_max_rel_err(_np(y), ref) <= TOL_F32

    m, K, n = 64, 128, 128
    xa, wa = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=42, w_layout="nk")
    dy, _ = gen.ag_inputs(N, N * m, n, 1, gen.NORMAL1, gen.NORMAL002, seed=43)
    pb = dbg.Plan(N, 1, "uni")
    wsb = _ws(pb.backward_pair_workspace_size(m, K, n))
    dx = torch.empty(N, m, K, device=DEV)
    dw = torch.empty(N, n, K, device=DEV)
    dbg.cm_backward_pair(pb, xa.to(DEV), wa.to(DEV), dy.to(DEV), dx, dw, wsb)
    st, info = dbg.cm_check_status(wsb)
    assert st == 0, (st, info)
    assert oracle.normwise_max_rel_err(_np(dw), oracle.wgrad(gen.bf16_bits(xa), gen.bf16_bits(dy))) <= TOL_F32

    q, b = 2, 128
    a, _ = gen.ag_inputs(q * q, b, b, 1, gen.NORMAL1, gen.NORMAL002, seed=44)
    pc = dbg.Plan(q * q, 1, "uni")
    wsc = _ws(pc.cannon_workspace_size(b, b, b))
    c = torch.empty(q * q, b, b, device=DEV)
    bblk, _ = gen.ag_inputs(q * q, b, b, 1, gen.NORMAL1, gen.NORMAL002, seed=45)
    dbg.cm_cannon_gemm(pc, a.to(DEV), bblk.to(DEV), c, wsc, "nk")
    st, info = dbg.cm_check_status(wsc)
    assert st == 0, (st, info)


@pytest.mark.parametrize("epilogue", [1, 2, 3])
def test_planted_flag_index_is_reported(dbg, epilogue):
    N, M, k, n = 4, 1024, 128, 512
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=46, w_layout="nk")
    p = _plan(dbg, N, 1, "uni", CM_OPT_RS_EPILOGUE=epilogue, CM_OPT_TIMEOUT_NS=50_000_000)
    ids = N * p.steps(dbg.CM_OP_GEMM_RS) * 2       # the flag ids of the plan: (rank, step, stream)
    # the flag words are sized for the smaller (128-row) tiles of the two
    # kernels, so the pair kernel's indices leave them only past several
    # times the ids; 8 times moves every signal out (and, as bytes, still
    # inside the 2 MB of bucket buffers that follow)
    p.set_option(dbg.CM_OPT_DEBUG_FLAG_OFFSET, 8 * ids)
    _, (st, info) = _rs(dbg, p, x, w)
    assert st == dbg.CM_ERR_BOUNDS, (st, info)
    assert info[0] == dbg.CM_ERR_BOUNDS and info[3] == KSITE_BOUNDS_FLAG, info
    p.set_option(dbg.CM_OPT_DEBUG_FLAG_OFFSET, 0)
    y, (st, info) = _rs(dbg, p, x, w)
    assert st == 0, (st, info)
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    assert oracle.normwise_max_rel_err(_np(y), ref) <= TOL_F32
