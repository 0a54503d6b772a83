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
Every workspace starts filled with 0xFF bytes (NaN as bf16 and as fp32), so a
tile that reads a receive slot or a bucket before its producer wrote it
yields NaN and fails (the ordering hazards of "Hiding Tensor-Parallel
Collectives: AG/RS Overlap in Megatron", sections 5 and 7: nothing is read
before its producer has written it).

Full-size workloads: the Megatron-SP fc1 and fc2 layers and the GPT-3 layer
are compared with the oracle in full; the MLP sweep on rows the oracle
computes one by one -- at least one in every 128-row block of every (rank,
shard) pair for AllGather->GEMM and of every bucket for GEMM->ReduceScatter,
so every CTA half of every pair tile of every task, for every chunk count,
is compared element by element -- and in full against torch.matmul on the
concatenated operands on the device (a second, independent computation).
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
    ws = torch.full((plan.ag_workspace_size(m, K),), 0xFF, dtype=torch.uint8, device=DEV)
    y = torch.full((N, N * m, n), float("nan"), dtype=ydtype, device=DEV)
    cm.cm_ag_gemm(plan, x.to(DEV), w.to(DEV), y, ws, layout)
    st, info = cm.cm_check_status(ws)
    if check:
        assert st == 0, f"status {st} info {info}"
    return y, st, info


def run_rs(plan, x, w, layout="nk", ydtype=torch.float32, check=True):
    N, M, k = x.shape
    n = w.shape[1] if layout == "nk" else w.shape[2]
    ws = torch.full((plan.rs_workspace_size(M, n),), 0xFF, dtype=torch.uint8, device=DEV)
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


# ---- full-size workloads ----------------------------------------------------------

BLOCK = 128   # rows of one CTA's half of a 256-row pair tile


def _block_rows(rows, rng):
    """One random row in every BLOCK-row block of [0, rows), plus the first and last row."""
    out = [b + int(rng.integers(0, min(BLOCK, rows - b))) for b in range(0, rows, BLOCK)]
    return sorted(set(out) | {0, rows - 1})


def _ag_rows(N, m, rng):
    """(rank, gathered row) samples: for every (rank r, shard j) pair, one row
    in every 128-row block of the shard (and its first and last row).  Every
    task (r, j) of every ring schedule writes rows j*m.. of Y_r, and every CTA
    half of every pair tile of that task covers one such block, whatever the
    chunk count (chunks are multiples of 128 rows here)."""
    ranks, rows = [], []
    for r in range(N):
        for j in range(N):
            for i in _block_rows(m, rng):
                ranks.append(r)
                rows.append(j * m + i)
    return np.array(ranks), np.array(rows)


def _rs_rows(N, Mb, rng):
    """(owner, row) samples: one row in every 128-row block of every bucket
    (and its first and last row) -- every chunk and pair-tile half of every
    bucket, each of which is the sum of every rank's contribution."""
    owners, rows = [], []
    for o in range(N):
        for i in _block_rows(Mb, rng):
            owners.append(o)
            rows.append(i)
    return np.array(owners), np.array(rows)


def _torch_ag(x, w, layout="nk"):
    """Y_r = concat_j(X_j) @ W_r by torch.matmul (cuBLAS, bf16 in, fp32 accumulate), on the device."""
    N, m, K = x.shape
    X = x.reshape(N * m, K)
    return torch.stack([X @ (w[r].t() if layout == "nk" else w[r]) for r in range(N)])


def _torch_rs(x, w, layout="nk"):
    """sum_r X_r @ W_r as one torch.matmul over the contraction-concatenated operands."""
    N, M, k = x.shape
    X = x.permute(1, 0, 2).reshape(M, N * k)
    W = (w.transpose(1, 2) if layout == "nk" else w).reshape(N * k, -1)
    return (X @ W).reshape(N, M // N, -1)


def _check_ag_full(N, m, K, n, direction, chunks, seed, layout="nk", full_oracle=False):
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=seed, w_layout=layout)
    y, _, _ = run_ag(cm.Plan(N, chunks, direction), x, w, layout, torch.bfloat16)
    assert torch.isfinite(y).all()
    xd, wd = x.to(DEV), w.to(DEV)
    assert _err(y, _np(_torch_ag(xd, wd, layout))) <= TOL
    if full_oracle:
        ref = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), layout)
        assert _err(y, ref) <= TOL
        return
    ranks, rows = _ag_rows(N, m, np.random.default_rng(seed))
    ref = oracle.ag_gemm_rows(gen.bf16_bits(x), gen.bf16_bits(w), ranks, rows, layout)
    got = y[torch.as_tensor(ranks, device=DEV), torch.as_tensor(rows, device=DEV)]
    assert oracle.normwise_max_rel_err(_np(got), ref) <= TOL


def _check_rs_full(N, M, k, n, direction, chunks, seed, layout="nk", full_oracle=False):
    x, w = gen.rs_inputs(N, M, k, n, gen.NORMAL1, gen.NORMAL002, seed=seed, w_layout=layout)
    y, _, _ = run_rs(cm.Plan(N, chunks, direction), x, w, layout, torch.bfloat16)
    assert torch.isfinite(y).all()
    xd, wd = x.to(DEV), w.to(DEV)
    assert _err(y, _np(_torch_rs(xd, wd, layout))) <= TOL
    if full_oracle:
        ref = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), layout)
        assert _err(y, ref) <= TOL
        return
    owners, rows = _rs_rows(N, M // N, np.random.default_rng(seed))
    ref = oracle.gemm_rs_rows(gen.bf16_bits(x), gen.bf16_bits(w), owners, rows, layout)
    got = y[torch.as_tensor(owners, device=DEV), torch.as_tensor(rows, device=DEV)]
    assert oracle.normwise_max_rel_err(_np(got), ref) <= TOL


def test_sp_mlp_fc1_ag_n8():
    """Megatron-SP MLP fc1 AllGather->GEMM, every output element against the oracle."""
    a = gen.WORKLOADS["sp_mlp_fc1_ag_n8"]["ag"]
    _check_ag_full(8, a["m"], a["K"], a["n"], "uni", 1, a["seed"], full_oracle=True)


def test_sp_mlp_fc2_rs_n8():
    """Megatron-SP MLP fc2 GEMM->ReduceScatter, every output element against the oracle."""
    r = gen.WORKLOADS["sp_mlp_fc2_rs_n8"]["rs"]
    _check_rs_full(8, r["M"], r["k"], r["n"], "uni", 1, r["seed"], full_oracle=True)


def test_gpt3_layer_bidi():
    """GPT-3 layer (QKV AllGather->GEMM, attention-out GEMM->ReduceScatter),
    bidirectional ring, every output element against the oracle."""
    wl = gen.WORKLOADS["gpt3_h12288_s2048_n8"]
    a, r = wl["ag"], wl["rs"]
    _check_ag_full(8, a["m"], a["K"], a["n"], "bidi", 1, a["seed"], full_oracle=True)
    _check_rs_full(8, r["M"], r["k"], r["n"], "bidi", 1, r["seed"], full_oracle=True)


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
    owners, orow = _rs_rows(N, r["M"] // N, rng)
    ref_r = oracle.gemm_rs_rows(gen.bf16_bits(xr), gen.bf16_bits(wr), owners, orow, "nk")
    return dict(xa=xa, wa=wa, xr=xr, wr=wr, ranks=ranks, rows=rows, ref_a=ref_a, owners=owners, orow=orow,
                ref_r=ref_r)


@functools.lru_cache(maxsize=1)
def _mlp_torch(N):
    """torch.matmul results of the MLP sweep at N ranks (every element), on the device."""
    c = _mlp_case(N)
    return _torch_ag(c["xa"].to(DEV), c["wa"].to(DEV)), _torch_rs(c["xr"].to(DEV), c["wr"].to(DEV))


SWEEP = [(N, c, d) for N in (4, 8, 16) for d in ("uni", "bidi") for c in (1, 2, 4)]


@pytest.mark.parametrize("N,chunks,direction", SWEEP)
def test_mlp_h8192_sweep_points(N, chunks, direction):
    """Every (N, chunks, ring) point of the MLP h=8192, ffn=28672, s=8192
    chunk/ring sweep, both ops at full size: the oracle's rows in every
    128-row block of every task, and every element against torch.matmul."""
    c = _mlp_case(N)
    t_ag, t_rs = _mlp_torch(N)
    y, _, _ = run_ag(cm.Plan(N, chunks, direction), c["xa"], c["wa"], "nk", torch.bfloat16)
    assert torch.isfinite(y).all()
    got = y[torch.as_tensor(c["ranks"], device=DEV), torch.as_tensor(c["rows"], device=DEV)]
    assert oracle.normwise_max_rel_err(_np(got), c["ref_a"]) <= TOL
    assert ((y.float() - t_ag.float()).abs().max() / t_ag.float().abs().max()).item() <= TOL
    del y
    y, _, _ = run_rs(cm.Plan(N, chunks, direction), c["xr"], c["wr"], "nk", torch.bfloat16)
    assert torch.isfinite(y).all()
    got = y[torch.as_tensor(c["owners"], device=DEV), torch.as_tensor(c["orow"], device=DEV)]
    assert oracle.normwise_max_rel_err(_np(got), c["ref_r"]) <= TOL
    assert ((y.float() - t_rs.float()).abs().max() / t_rs.float().abs().max()).item() <= TOL
