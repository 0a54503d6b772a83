"""GEMM->ReduceScatter with the received partial bucket preloaded into the
tile's tensor-memory accumulator (CM_OPT_RS_PRELOAD = 1: all of it; 3: half,
the rest added in the epilogue): the same result as the epilogue-add path
(0), against the oracle, exactly on integer inputs, and at the full MLP
sweep size on sampled rows.  The automatic choice (2, the default) picks one
of the first two by the tile's K-slice count; it is checked against both.
The preload applies to buckets in per-step buffers (CM_OPT_RS_IN_PLACE = 0),
which every test here uses."""

import numpy as np
import pytest
import torch

import oracle
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen
from test_gpu_parity import TOL, TOL_F32, _np, run_rs

pytestmark = pytest.mark.gpu


def _plan(N, chunks, direction, preload, kernel=0):
    p = cm.Plan(N, chunks, direction)
    p.set_option(cm.CM_OPT_KERNEL, kernel)
    p.set_option(cm.CM_OPT_RS_PRELOAD, preload)
    p.set_option(cm.CM_OPT_RS_IN_PLACE, 0)   # the preload reads per-step bucket buffers
    return p


@pytest.mark.parametrize("N,M,k,n,chunks,direction", [
    (2, 128, 256, 512, 1, "uni"),       # bucket rows below one CTA's 128
    (3, 600, 200, 296, 2, "bidi"),      # ragged rows / columns / K; the owner adds a second partial
    (4, 1536, 320, 768, 1, "uni"),      # row tiles straddling the pair split; 3 column tiles
    (8, 2048, 192, 1032, 4, "uni"),     # 64-row chunks, ragged last column tile
    (5, 1360, 72, 520, 1, "bidi"),      # odd rank count both ways, one K slice
])
@pytest.mark.parametrize("layout", ["nk", "kn"])
@pytest.mark.parametrize("ydtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("mode", [1, 3])
def test_preload_vs_oracle(N, M, k, n, chunks, direction, layout, ydtype, mode):
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=M + k, w_layout=layout)
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), layout)
    y, _, _ = run_rs(_plan(N, chunks, direction, mode), x, w, layout, ydtype)
    e = oracle.normwise_max_rel_err(_np(y), ref)
    assert np.isfinite(_np(y)).all()
    assert e <= (TOL_F32 if ydtype == torch.float32 else TOL), e


@pytest.mark.parametrize("direction", ["uni", "bidi"])
@pytest.mark.parametrize("mode", [1, 3])
def test_preload_exact_on_integers(direction, mode):
    """Small-integer inputs keep every fp32 partial sum exact, so both paths
    and the oracle agree bit for bit whatever the summation order."""
    N, M, k, n = 6, 1536, 256, 640
    g = torch.Generator().manual_seed(5)
    x = torch.randint(-3, 4, (N, M, k), generator=g).to(torch.bfloat16)
    w = torch.randint(-2, 3, (N, n, k), generator=g).to(torch.bfloat16)
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    y1, _, _ = run_rs(_plan(N, 2, direction, mode), x, w, "nk")
    y0, _, _ = run_rs(_plan(N, 2, direction, 0), x, w, "nk")
    assert np.array_equal(_np(y1), ref)
    assert torch.equal(y1, y0)


def test_preload_matches_epilogue_add_and_repeats():
    """Two calls in a row on one workspace give identical bits; the result
    differs from the epilogue-add path only by fp32 summation order."""
    N, M, k, n = 8, 4096, 512, 1024
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=11, w_layout="nk")
    p1 = _plan(N, 1, "uni", 1)
    dev = "cuda:0"
    ws = torch.full((p1.rs_workspace_size(M, n),), 0xFF, dtype=torch.uint8, device=dev)
    xd, wd = x.to(dev), w.to(dev)
    ya = torch.empty(N, M // N, n, dtype=torch.float32, device=dev)
    yb = torch.empty_like(ya)
    cm.cm_gemm_rs(p1, xd, wd, ya, ws, "nk")
    cm.cm_gemm_rs(p1, xd, wd, yb, ws, "nk")
    assert cm.cm_check_status(ws)[0] == 0
    assert torch.equal(ya, yb)
    y0, _, _ = run_rs(_plan(N, 1, "uni", 0), x, w, "nk")
    assert (ya - y0).abs().max().item() <= 1e-4 * y0.abs().max().item()


@pytest.mark.parametrize("k,picked", [(256, 1), (512, 1), (1024, 0), (4096, 0)])
def test_automatic_choice_matches_the_path_it_picks(k, picked):
    """The default (automatic) setting gives the bits of the path it picks:
    all preloaded for at most 8 K slices, none beyond."""
    N, M, n = 4, 2048, 512
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=k, w_layout="nk")
    p = cm.Plan(N, 1, "uni")
    p.set_option(cm.CM_OPT_RS_IN_PLACE, 0)   # default preload option, per-step buffers
    auto, _, _ = run_rs(p, x, w, "nk")
    y, _, _ = run_rs(_plan(N, 1, "uni", picked), x, w, "nk")
    assert torch.equal(auto, y)


def test_preload_skipped_signal_times_out():
    """A dropped done-signal now stalls the tile scheduler (which waits for
    the bucket before loading it): the bounded wait reports a timeout and the
    context stays usable."""
    N, M, k, n = 4, 1024, 256, 512
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=3, w_layout="nk")
    p = _plan(N, 1, "uni", 1)
    p.set_option(cm.CM_OPT_TIMEOUT_NS, 50_000_000)
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, (cm.CM_OP_GEMM_RS << 16) | (1 << 8) | 0)
    _, st, info = run_rs(p, x, w, "nk", check=False)
    assert st == cm.CM_ERR_TIMEOUT, (st, info)
    y, _, _ = run_rs(_plan(N, 1, "uni", 1), x, w, "nk")   # the next call works
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    assert oracle.normwise_max_rel_err(_np(y), ref) <= TOL_F32


@pytest.mark.parametrize("N,mode", [(8, 1), (16, 3)])
def test_preload_full_size_sampled(N, mode):
    """The MLP h=8192, ffn=28672, s=8192 fc2 GEMM-RS at full size, sampled rows."""
    s = gen.mlp_shapes(N)["rs"]
    wl = gen.WORKLOADS["mlp_h8192_ffn28672_s8192"]["rs"]
    x, w = gen.rs_inputs(N, s["M"], s["k"], s["n"], wl["x"], wl["w"], wl["seed"], "nk")
    y, _, _ = run_rs(_plan(N, 1, "uni", mode), x, w, "nk", torch.bfloat16)
    Mb = s["M"] // N
    rng = np.random.default_rng(N)
    pairs = [(o, r) for o in range(N) for r in (0, 255, 256, Mb - 1)]
    pairs += [(int(o), int(r)) for o, r in zip(rng.integers(0, N, 16), rng.integers(0, Mb, 16))]
    owners = np.array([o for o, _ in pairs], dtype=np.int32)
    rows = np.array([r for _, r in pairs], dtype=np.int64)
    ref = oracle.gemm_rs_rows(gen.bf16_bits(x), gen.bf16_bits(w), owners, rows, "nk")
    got = _np(y)[owners, rows]
    assert oracle.normwise_max_rel_err(got, ref) <= TOL
