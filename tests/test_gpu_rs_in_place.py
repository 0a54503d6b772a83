"""GEMM->ReduceScatter with every bucket accumulated in place (one fp32
buffer per bucket and ring stream; each contributor after the first adds its
partial product into it where it lies, with a TMA reduce-add at L2 on the
CTA-pair kernel) against the oracle and against the per-step buffers
(CM_OPT_RS_IN_PLACE = 0, where each rank loads the partial bucket, adds and
stores a new one).

The ring order of the additions is the same in both ("Overlap Communication
with Dependent Computation via Decomposition in Large Deep Learning Models",
section "The idea", Einsum -> ReduceScatter: each rank adds its contribution
to the bucket it received, in ring order), and so is every fp32 addition:
bucket + partial, one rounding each.  With the received bucket added in the
epilogue on both sides (no preload into tensor memory), the fp32 outputs
must therefore be identical bit for bit.  Workspaces start as 0xFF bytes
(NaN), so an addition into a bucket that its first contributor had not yet
written, or a read by the owner before the last addition, shows up as NaN.
"""

import numpy as np
import pytest
import torch

import oracle
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen
from test_gpu_parity import TOL, TOL_F32, _np, run_rs

pytestmark = pytest.mark.gpu

PAIR, SINGLE = 0, 1


def _plan(N, chunks, direction, in_place, kernel=PAIR, preload=0, epilogue=0):
    p = cm.Plan(N, chunks, direction)
    p.set_option(cm.CM_OPT_RS_IN_PLACE, in_place)
    p.set_option(cm.CM_OPT_KERNEL, kernel)
    p.set_option(cm.CM_OPT_RS_PRELOAD, preload)
    p.set_option(cm.CM_OPT_RS_EPILOGUE, epilogue)
    return p


# the CTA-pair kernel with each RS epilogue (TMA copies / two warp groups
# with vector adds / every warp with vector adds), and the single-CTA kernel
KERNEL_EPILOGUES = [(PAIR, 1), (PAIR, 2), (PAIR, 3), (SINGLE, 0)]


@pytest.mark.parametrize("kernel,epilogue", KERNEL_EPILOGUES)
@pytest.mark.parametrize("N,M,k,n,chunks,direction", [
    (2, 256, 128, 512, 1, "uni"),
    (3, 768, 200, 296, 2, "uni"),       # ragged k and n
    (4, 2048, 320, 768, 2, "bidi"),     # even N: the counter-clockwise stream is one hop shorter
    (5, 1280, 136, 520, 1, "bidi"),     # odd N: both streams equally long
    (8, 4096, 256, 1024, 4, "uni"),     # chunks of 128 rows: two chunks per pair tile
    (8, 2048, 64, 256, 1, "bidi"),
    (4, 1536, 96, 1032, 1, "uni"),      # ragged last column tile, rows straddling the pair split
])
def test_in_place_matches_per_step_buffers_bitwise(kernel, epilogue, N, M, k, n, chunks, direction):
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=N * 100 + k, w_layout="nk")
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    y0, _, _ = run_rs(_plan(N, chunks, direction, 0, kernel, 0, epilogue), x, w, "nk", torch.float32)
    y1, _, _ = run_rs(_plan(N, chunks, direction, 1, kernel, 0, epilogue), x, w, "nk", torch.float32)
    assert torch.isfinite(y1).all()
    assert oracle.normwise_max_rel_err(_np(y1), ref) <= TOL_F32
    assert torch.equal(y0, y1)


@pytest.mark.parametrize("in_place", [1, 0])
@pytest.mark.parametrize("preload", [0, 1, 3])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
def test_rs_epilogues_agree_bitwise(in_place, preload, direction):
    """The CTA-pair RS epilogues make the same fp32 additions in the same
    order: the same bits, in both bucket modes and every preload mode."""
    N, M, k, n = 8, 2048, 256, 1288
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=71, w_layout="nk")
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    ys = {}
    for epilogue in (1, 2, 3):
        for ydtype in (torch.float32, torch.bfloat16):
            y, _, _ = run_rs(_plan(N, 2, direction, in_place, PAIR, preload, epilogue), x, w, "nk", ydtype)
            assert oracle.normwise_max_rel_err(_np(y), ref) <= (TOL_F32 if ydtype == torch.float32 else TOL)
            ys[epilogue, ydtype] = y
    for ydtype in (torch.float32, torch.bfloat16):
        assert torch.equal(ys[1, ydtype], ys[2, ydtype]) and torch.equal(ys[1, ydtype], ys[3, ydtype])


@pytest.mark.parametrize("preload", [0, 1, 2, 3])
def test_in_place_with_owner_preload(preload):
    """Only the owner's tile reads its bucket, and only there does the
    preload apply; every preload mode gives the oracle's result."""
    N, M, k, n = 8, 4096, 256, 2048
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=91, w_layout="kn")
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "kn")
    for direction in ("uni", "bidi"):
        y, _, _ = run_rs(_plan(N, 1, direction, 1, PAIR, preload), x, w, "kn", torch.float32)
        assert oracle.normwise_max_rel_err(_np(y), ref) <= TOL_F32
        yb, _, _ = run_rs(_plan(N, 1, direction, 1, PAIR, preload), x, w, "kn", torch.bfloat16)
        assert oracle.normwise_max_rel_err(_np(yb), ref) <= TOL


def test_in_place_exact_on_integers():
    """Small integers: every partial and every sum is exact in fp32, so the
    output equals the oracle exactly, for both kernels and both rings."""
    N, M, k, n = 4, 1024, 96, 640
    g = torch.Generator().manual_seed(12)
    x = torch.randint(-3, 4, (N, M, k), generator=g).to(torch.bfloat16)
    w = torch.randint(-3, 4, (N, n, k), generator=g).to(torch.bfloat16)
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    for kernel, epilogue in KERNEL_EPILOGUES:
        for direction in ("uni", "bidi"):
            y, _, _ = run_rs(_plan(N, 2, direction, 1, kernel, 2, epilogue), x, w, "nk", torch.float32)
            assert np.array_equal(_np(y), ref)


@pytest.mark.parametrize("epilogue", [1, 2, 3])
@pytest.mark.parametrize("in_place", [1, 0])
def test_in_place_dropped_signal_times_out(epilogue, in_place):
    """A contributor that never signals: its successor's addition (or load)
    and the owner's read wait for it, time out, and the next call is
    correct, with buckets in place and with per-step buffers."""
    N, M, k, n = 4, 1024, 128, 256
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=5, w_layout="nk")
    p = _plan(N, 1, "uni", in_place, PAIR, 0, epilogue)
    p.set_option(cm.CM_OPT_TIMEOUT_NS, 50_000_000)
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, (cm.CM_OP_GEMM_RS << 16) | (1 << 8) | 1)
    _, st, info = run_rs(p, x, w, "nk", torch.float32, check=False)
    assert st == cm.CM_ERR_TIMEOUT, (st, info)
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, -1)
    y, _, _ = run_rs(p, x, w, "nk", torch.float32)
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    assert oracle.normwise_max_rel_err(_np(y), ref) <= TOL_F32


def test_in_place_back_to_back_on_one_workspace():
    """Calls that share a workspace on one stream: each call's first
    contributor overwrites the previous call's bucket before anyone adds."""
    N, M, k, n = 8, 2048, 192, 768
    sets = [gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=s, w_layout="nk") for s in (31, 32)]
    refs = [oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk") for x, w in sets]
    p = _plan(N, 2, "uni", 1)
    dev = "cuda:0"
    ws = torch.full((p.rs_workspace_size(M, n),), 0xFF, dtype=torch.uint8, device=dev)
    outs = [torch.full((N, M // N, n), float("nan"), device=dev) for _ in sets]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for (x, w), y in zip(sets, outs):
            cm.cm_gemm_rs(p, x.to(dev), w.to(dev), y, ws, "nk", s)
    st, info = cm.cm_check_status(ws, s)
    assert st == 0, (st, info)
    for y, ref in zip(outs, refs):
        assert oracle.normwise_max_rel_err(_np(y), ref) <= TOL_F32


@pytest.mark.parametrize("direction", ["uni", "bidi"])
@pytest.mark.parametrize("N,chunks", [(4, 1), (8, 2), (5, 1)])
def test_task_orders_agree_bitwise(N, chunks, direction):
    """The ring's own task order (rank-blocked one-way, stream-blocked
    two-way) and the step-major one only reorder the tiles: every
    output element is the same dot product (AllGather->GEMM) or the same
    ring-ordered fp32 sum (GEMM->ReduceScatter), so the bits agree."""
    m, K, n = 256, 384, 768
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=61, w_layout="nk")
    xr, wr = gen.rs_inputs(N, N * m, K, n, gen.NORMAL1, gen.NORMAL002, seed=62, w_layout="nk")
    from test_gpu_parity import run_ag
    outs = []
    for order in (1, 2):
        p = cm.Plan(N, chunks, direction)
        p.set_option(cm.CM_OPT_TASK_ORDER, order)
        y, _, _ = run_ag(p, x, w, "nk", torch.float32)
        yr, _, _ = run_rs(p, xr, wr, "nk", torch.float32)
        outs.append((y, yr))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
    ref = oracle.gemm_rs(gen.bf16_bits(xr), gen.bf16_bits(wr), "nk")
    assert oracle.normwise_max_rel_err(_np(outs[1][1]), ref) <= TOL_F32


@pytest.mark.parametrize("kernel,epilogue", KERNEL_EPILOGUES)
@pytest.mark.parametrize("N,M,k,n,chunks,direction,slabs", [
    (4, 1024, 128, 1024, 1, "uni", 2),
    (8, 4096, 256, 2048, 4, "uni", 4),      # chunk pairs
    (5, 1280, 136, 1536, 1, "bidi", 3),     # odd N, three slabs of two column tiles
    (4, 2048, 320, 1032, 2, "bidi", 2),     # ragged last column tile: the count falls back to a divisor
])
@pytest.mark.parametrize("in_place", [1, 0])
def test_column_slabs_agree_bitwise(kernel, epilogue, N, M, k, n, chunks, direction, slabs, in_place):
    """CM_OPT_RS_COL_SLABS only reorders the tiles: every bucket tile gets
    the same additions in the same ring order, so the bits agree with one
    pass, and with the oracle within the fp32 bar, for buckets in place and
    for per-step buffers."""
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=N * 7 + slabs, w_layout="nk")
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    p1 = _plan(N, chunks, direction, in_place, kernel, 0, epilogue)
    p1.set_option(cm.CM_OPT_RS_COL_SLABS, 1)
    y1, _, _ = run_rs(p1, x, w, "nk", torch.float32)
    ps = _plan(N, chunks, direction, in_place, kernel, 0, epilogue)
    ps.set_option(cm.CM_OPT_RS_COL_SLABS, slabs)
    ys, _, _ = run_rs(ps, x, w, "nk", torch.float32)
    assert torch.isfinite(ys).all()
    assert oracle.normwise_max_rel_err(_np(ys), ref) <= TOL_F32
    assert torch.equal(y1, ys)


@pytest.mark.parametrize("epilogue", [1, 2, 3])
@pytest.mark.parametrize("hint", [0, 1, 2])
def test_bucket_l2_hints_keep_the_bits(epilogue, hint):
    """CM_OPT_RS_BUCKET_HINT changes only the L2 policy of the TMA
    epilogue's bucket writes and adds (the vector epilogues take none): the
    same bits as with no policy (3)."""
    N, M, k, n = 8, 2048, 192, 1032
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=hint * 10 + epilogue, w_layout="nk")
    p0 = _plan(N, 2, "uni", 1, PAIR, 0, epilogue)
    p0.set_option(cm.CM_OPT_RS_BUCKET_HINT, 3)
    y0, _, _ = run_rs(p0, x, w, "nk", torch.float32)
    p = _plan(N, 2, "uni", 1, PAIR, 0, epilogue)
    p.set_option(cm.CM_OPT_RS_BUCKET_HINT, hint)
    y1, _, _ = run_rs(p, x, w, "nk", torch.float32)
    assert torch.equal(y0, y1)
