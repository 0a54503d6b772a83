"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bars (the arithmetic is bf16 products accumulated in fp32):
* normwise max relative error  max|y - ref| / max|ref|  <= 2e-2 for every
  output tensor (the stated bound for bf16 inputs / fp32 accumulation);
* fp32 outputs additionally <= 1e-4: an fp32 sum of K exact bf16 products
  differs from the exact sum by at most about K * 2^-24 * sum|a*b|, far below;
* placement is bit-exact: tagged inputs make every output an exact small
  integer that names its source shard and row;
* AllGather->GEMM is bit-identical across chunk counts, ring directions, the
  step-serial mode and the undecomposed path (each output element is the same
  tensor-core dot product whichever tile computes it).
Full-size workloads are checked on sampled rows the oracle computes one by one.
"""

import functools

import numpy as np
import pytest
import torch

import oracle
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

TOL = 2e-2
TOL_F32 = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


DEV = "cuda:0"


def run_ag(plan, x, w, layout="nk", ydtype=torch.float32, check=True):
    N, m, K = x.shape
    n = w.shape[1] if layout == "nk" else w.shape[2]
    ws = torch.empty(plan.ag_workspace_size(m, K), dtype=torch.uint8, device=DEV)
    y = torch.full((N, N * m, n), float("nan"), dtype=ydtype, device=DEV)
    cm.cm_ag_gemm(plan, x.to(DEV), w.to(DEV), y, ws, layout)
    st, info = cm.cm_check_status(ws)
    if check:
        assert st == 0, f"status {st} info {info}"
    return y, st, info


def run_rs(plan, x, w, layout="nk", ydtype=torch.float32, check=True):
    N, M, k = x.shape
    n = w.shape[1] if layout == "nk" else w.shape[2]
    ws = torch.empty(plan.rs_workspace_size(M, n), dtype=torch.uint8, device=DEV)
    y = torch.full((N, M // N, n), float("nan"), dtype=ydtype, device=DEV)
    cm.cm_gemm_rs(plan, x.to(DEV), w.to(DEV), y, ws, layout)
    st, info = cm.cm_check_status(ws)
    if check:
        assert st == 0, f"status {st} info {info}"
    return y, st, info


def _np(y):
    return y.detach().float().cpu().double().numpy()


def _err(y, ref):
    return oracle.normwise_max_rel_err(_np(y) if torch.is_tensor(y) else y, ref)


def _assert_close(y, ref, ydtype):
    e = _err(y, ref)
    assert np.isfinite(_np(y)).all()
    assert e <= TOL, e
    if ydtype == torch.float32:
        assert e <= TOL_F32, e


# ---- small workloads, full oracle --------------------------------------------

@pytest.mark.parametrize("direction", ["uni", "bidi", "none"])
@pytest.mark.parametrize("chunks", [1, 2])
@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_tiny_n2_full(direction, chunks, layout):
    wl = gen.WORKLOADS["tiny_n2"]
    N, a, r = wl["N"], wl["ag"], wl["rs"]
    x, w = gen.ag_inputs(N, a["m"], a["K"], a["n"], a["x"], a["w"], a["seed"], layout)
    ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), layout)
    plan = cm.Plan(N, chunks, direction)
    y, _, _ = run_ag(plan, x, w, layout)
    _assert_close(y, ref, torch.float32)
    xr, wr = gen.rs_inputs(N, r["M"], r["k"], r["n"], r["x"], r["w"], r["seed"], layout)
    refr = oracle.gemm_rs(gen.bf16_bits(xr), gen.bf16_bits(wr), layout)
    yr, _, _ = run_rs(plan, xr, wr, layout)
    _assert_close(yr, refr, torch.float32)


@pytest.mark.parametrize("N,m,K,n", [(3, 200, 200, 296), (5, 136, 72, 520), (2, 264, 1032, 264)])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
@pytest.mark.parametrize("chunks", [1, 2])
@pytest.mark.parametrize("ydtype", [torch.float32, torch.bfloat16])
def test_ragged_multi_tile(N, m, K, n, direction, chunks, ydtype):
    """Several row / column tiles, ragged tails in rows, columns and K."""
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=N * 31 + m, w_layout="nk")
    ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    plan = cm.Plan(N, chunks, direction)
    y, _, _ = run_ag(plan, x, w, "nk", ydtype)
    _assert_close(y, ref, ydtype)
    xr, wr = gen.rs_inputs(N, N * m, K, n, gen.NORMAL1, gen.NORMAL002, seed=N * 37 + m, w_layout="nk")
    refr = oracle.gemm_rs(gen.bf16_bits(xr), gen.bf16_bits(wr), "nk")
    yr, _, _ = run_rs(plan, xr, wr, "nk", ydtype)
    _assert_close(yr, refr, ydtype)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
def test_tagged_placement_bit_exact(N, direction):
    m, K, n = 160, 64, 256
    x, w = gen.tagged_ag_inputs(N, m, K, n, "nk")
    ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    for ydtype in (torch.float32, torch.bfloat16):
        y, _, _ = run_ag(cm.Plan(N, 2 if N % 2 == 0 else 1, direction), x, w, "nk", ydtype)
        assert np.array_equal(_np(y), ref)


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_n1_is_plain_gemm(layout):
    x, w = gen.ag_inputs(1, 384, 512, 768, gen.NORMAL1, gen.NORMAL002, seed=5, w_layout=layout)
    ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), layout)
    for d in ("uni", "bidi", "none"):
        y, _, _ = run_ag(cm.Plan(1, 1, d), x, w, layout)
        _assert_close(y, ref, torch.float32)
    xr, wr = gen.rs_inputs(1, 384, 512, 768, gen.NORMAL1, gen.NORMAL002, seed=6, w_layout=layout)
    refr = oracle.gemm_rs(gen.bf16_bits(xr), gen.bf16_bits(wr), layout)
    yr, _, _ = run_rs(cm.Plan(1, 1, "uni"), xr, wr, layout)
    _assert_close(yr, refr, torch.float32)


def test_ag_invariant_to_schedule_bitwise():
    N, m, K, n = 4, 256, 512, 512
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=77, w_layout="nk")
    base, _, _ = run_ag(cm.Plan(N, 1, "none"), x, w, "nk", torch.float32)
    variants = [(1, "uni"), (2, "uni"), (4, "uni"), (1, "bidi"), (2, "bidi")]
    for chunks, d in variants:
        y, _, _ = run_ag(cm.Plan(N, chunks, d), x, w, "nk", torch.float32)
        assert torch.equal(y, base), (chunks, d)
    p = cm.Plan(N, 2, "uni")
    p.set_option(cm.CM_OPT_SERIAL_STEPS, 1)
    y, _, _ = run_ag(p, x, w, "nk", torch.float32)
    assert torch.equal(y, base)
    p = cm.Plan(N, 1, "bidi")
    p.set_option(cm.CM_OPT_GRID, 7)      # few CTAs: many tiles per CTA
    y, _, _ = run_ag(p, x, w, "nk", torch.float32)
    assert torch.equal(y, base)


def test_weight_layouts_agree():
    N, m, K, n = 3, 128, 256, 512
    x, w_nk = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=9, w_layout="nk")
    w_kn = w_nk.transpose(1, 2).contiguous()
    a, _, _ = run_ag(cm.Plan(N, 1, "uni"), x, w_nk, "nk")
    b, _, _ = run_ag(cm.Plan(N, 1, "uni"), x, w_kn, "kn")
    assert torch.equal(a, b)


def test_rs_schedules_agree():
    N, M, k, n = 4, 1024, 384, 768
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=11, w_layout="nk")
    ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    for chunks, d in [(1, "uni"), (2, "uni"), (4, "bidi"), (1, "none")]:
        y, _, _ = run_rs(cm.Plan(N, chunks, d), x, w, "nk", torch.float32)
        _assert_close(y, ref, torch.float32)
    p = cm.Plan(N, 2, "bidi")
    p.set_option(cm.CM_OPT_SERIAL_STEPS, 1)
    y, _, _ = run_rs(p, x, w, "nk", torch.float32)
    _assert_close(y, ref, torch.float32)


def test_allreduce_is_rs_then_ag_on_gpu():
    """Concatenating the GEMM->ReduceScatter buckets gives sum_r X_r @ W_r."""
    N, M, k, n = 4, 512, 256, 512
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=13, w_layout="nk")
    y, _, _ = run_rs(cm.Plan(N, 1, "uni"), x, w, "nk", torch.float32)
    x64 = torch.cat([x[r].double() for r in range(N)], dim=1)
    w64 = torch.cat([w[r].double().t() for r in range(N)], dim=0)
    full = (x64 @ w64).numpy()
    assert oracle.normwise_max_rel_err(_np(y.reshape(M, n)), full) <= TOL_F32


# ---- bounded waits: a signal that never comes is reported, not hung ------------

def test_skipped_signal_times_out_and_context_survives():
    N, m, K, n = 4, 128, 128, 256
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=3, w_layout="nk")
    p = cm.Plan(N, 1, "uni")
    p.set_option(cm.CM_OPT_TIMEOUT_NS, 50_000_000)     # 50 ms
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, (cm.CM_OP_AG_GEMM << 16) | (1 << 8) | 0)
    _, st, info = run_ag(p, x, w, "nk", check=False)
    assert st == cm.CM_ERR_TIMEOUT, (st, info)
    assert info[0] == cm.CM_ERR_TIMEOUT
    xr, wr = gen.rs_inputs(N, 512, 128, 256, gen.NORMAL1, gen.NORMAL002, seed=4, w_layout="nk")
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, (cm.CM_OP_GEMM_RS << 16) | (2 << 8) | 1)
    _, st, info = run_rs(p, xr, wr, "nk", check=False)
    assert st == cm.CM_ERR_TIMEOUT, (st, info)
    # the context is still usable and the next call is correct
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, -1)
    ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    y, _, _ = run_ag(p, x, w, "nk")
    _assert_close(y, ref, torch.float32)


# ---- full-size workloads, sampled rows -----------------------------------------

def _ag_rows(N, m, rng, extra=48):
    """(rank, gathered row) samples: every shard's first/last row, tile edges, random."""
    rows = []
    for j in range(N):
        for i in {0, m - 1, min(127, m - 1), min(128, m - 1), m // 2}:
            rows.append(j * m + i)
    rows += list(rng.integers(0, N * m, size=extra))
    ranks = list(rng.integers(0, N, size=len(rows)))
    ranks[:N] = list(range(N))
    return np.array(ranks), np.array(rows)


def _check_ag_full(N, m, K, n, direction, chunks, seed, layout="nk"):
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=seed, w_layout=layout)
    y, _, _ = run_ag(cm.Plan(N, chunks, direction), x, w, layout, torch.bfloat16)
    rng = np.random.default_rng(seed)
    ranks, rows = _ag_rows(N, m, rng)
    ref = oracle.ag_gemm_rows(gen.bf16_bits(x), gen.bf16_bits(w), ranks, rows, layout)
    got = y[torch.as_tensor(ranks, device=DEV), torch.as_tensor(rows, device=DEV)]
    assert oracle.normwise_max_rel_err(_np(got), ref) <= TOL
    assert torch.isfinite(y).all()


def _check_rs_full(N, M, k, n, direction, chunks, seed, layout="nk"):
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=seed, w_layout=layout)
    y, _, _ = run_rs(cm.Plan(N, chunks, direction), x, w, layout, torch.bfloat16)
    rng = np.random.default_rng(seed)
    Mb = M // N
    owners = np.concatenate([np.arange(N), np.arange(N), rng.integers(0, N, 24)])
    rows = np.concatenate([np.zeros(N, int), np.full(N, Mb - 1), rng.integers(0, Mb, 24)])
    ref = oracle.gemm_rs_rows(gen.bf16_bits(x), gen.bf16_bits(w), owners, rows, layout)
    got = y[torch.as_tensor(owners, device=DEV), torch.as_tensor(rows, device=DEV)]
    assert oracle.normwise_max_rel_err(_np(got), ref) <= TOL
    assert torch.isfinite(y).all()


def test_sp_mlp_fc1_ag_n8():
    a = gen.WORKLOADS["sp_mlp_fc1_ag_n8"]["ag"]
    _check_ag_full(8, a["m"], a["K"], a["n"], "uni", 1, a["seed"])


def test_sp_mlp_fc2_rs_n8():
    r = gen.WORKLOADS["sp_mlp_fc2_rs_n8"]["rs"]
    _check_rs_full(8, r["M"], r["k"], r["n"], "uni", 1, r["seed"])


def test_gpt3_layer_bidi():
    wl = gen.WORKLOADS["gpt3_h12288_s2048_n8"]
    a, r = wl["ag"], wl["rs"]
    _check_ag_full(8, a["m"], a["K"], a["n"], "bidi", 1, a["seed"])
    _check_rs_full(8, r["M"], r["k"], r["n"], "bidi", 1, r["seed"])


@functools.lru_cache(maxsize=1)
def _mlp_case(N):
    """Inputs of the MLP sweep at N ranks (they depend on N only) and the
    oracle's sampled reference rows, made once for all chunk counts and rings."""
    s = gen.mlp_shapes(N)
    a, r = s["ag"], s["rs"]
    xa, wa = gen.ag_inputs(N, a["m"], a["K"], a["n"], gen.NORMAL1, gen.NORMAL002, seed=5000 + N, w_layout="nk")
    xr, wr = gen.rs_inputs(N, r["M"], r["k"], r["n"], gen.NORMAL1, gen.NORMAL002, seed=5002 + N, w_layout="nk")
    rng = np.random.default_rng(5000 + N)
    ranks, rows = _ag_rows(N, a["m"], rng)
    ref_a = oracle.ag_gemm_rows(gen.bf16_bits(xa), gen.bf16_bits(wa), ranks, rows, "nk")
    Mb = r["M"] // N
    owners = np.concatenate([np.arange(N), np.arange(N), rng.integers(0, N, 24)])
    orow = np.concatenate([np.zeros(N, int), np.full(N, Mb - 1), rng.integers(0, Mb, 24)])
    ref_r = oracle.gemm_rs_rows(gen.bf16_bits(xr), gen.bf16_bits(wr), owners, orow, "nk")
    return dict(xa=xa, wa=wa, xr=xr, wr=wr, ranks=ranks, rows=rows, ref_a=ref_a, owners=owners, orow=orow,
                ref_r=ref_r)


SWEEP = [(N, c, d) for N in (4, 8, 16) for d in ("uni", "bidi") for c in (1, 2, 4)]


@pytest.mark.parametrize("N,chunks,direction", SWEEP)
def test_mlp_h8192_sweep_points(N, chunks, direction):
    """Every (N, chunks, ring) point of the MLP h=8192, ffn=28672, s=8192
    chunk/ring sweep, both ops at full size, on sampled rows."""
    c = _mlp_case(N)
    y, _, _ = run_ag(cm.Plan(N, chunks, direction), c["xa"], c["wa"], "nk", torch.bfloat16)
    got = y[torch.as_tensor(c["ranks"], device=DEV), torch.as_tensor(c["rows"], device=DEV)]
    assert oracle.normwise_max_rel_err(_np(got), c["ref_a"]) <= TOL
    assert torch.isfinite(y).all()
    del y
    y, _, _ = run_rs(cm.Plan(N, chunks, direction), c["xr"], c["wr"], "nk", torch.bfloat16)
    got = y[torch.as_tensor(c["owners"], device=DEV), torch.as_tensor(c["orow"], device=DEV)]
    assert oracle.normwise_max_rel_err(_np(got), c["ref_r"]) <= TOL
    assert torch.isfinite(y).all()
