"""Pins for the fp64 oracle: each check ties it to something other than itself.

* brute force on tiny integer inputs (exact, pure-Python int64 sums)
* closed forms (constant and tagged inputs)
* N = 1 reduces to a plain GEMM (numpy's float64 matmul, a library routine)
* AllReduce = ReduceScatter followed by AllGather ("Tensor Parallelism ->
  Communication Patterns"): the owner-ordered concatenation of the
  GEMM->ReduceScatter buckets equals sum_r X_r @ W_r, computed as one numpy
  matmul over the contraction-concatenated operands
* the rank-by-rank ring simulation ("Overlap Communication ... via
  Decomposition", section "Why it works": the decomposition is exact) equals
  the definition: bit-identical for AllGather, within 1e-12 for the reordered
  ReduceScatter sums, for every chunk count and both ring directions
* planted mistakes (wrong neighbour, dropped contribution, transposed
  operand, shifted placement) fail at least one of the pins above
"""

import itertools

import numpy as np
import pytest
import torch

import oracle
from oracle import ring
from collective_matmul_decomposition_gb300 import inputs as gen


def _f64(t):
    return oracle.bf16_to_f64(gen.bf16_bits(t))


def _w_kn(w_bits, layout):
    """[N][K][n] view of per-rank weights as plain python ints/floats."""
    return w_bits if layout == "kn" else np.swapaxes(w_bits, 1, 2)


def _brute_ag(x, w_kn):
    """Pure-Python exact sums: Y_r[j*m+i][c] = sum_k X_j[i][k] * W_r[k][c]."""
    N, m, K = x.shape
    n = w_kn.shape[2]
    y = np.zeros((N, N * m, n), dtype=np.int64)
    for r, j, i, c in itertools.product(range(N), range(N), range(m), range(n)):
        s = 0
        for k in range(K):
            s += int(x[j, i, k]) * int(w_kn[r, k, c])
        y[r, j * m + i, c] = s
    return y


def _brute_rs(x, w_kn):
    """Pure-Python exact sums: Y_o[i][c] = sum_r sum_k X_r[o*Mb+i][k] * W_r[k][c]."""
    N, M, k_ = x.shape
    n = w_kn.shape[2]
    Mb = M // N
    y = np.zeros((N, Mb, n), dtype=np.int64)
    for o, i, c in itertools.product(range(N), range(Mb), range(n)):
        s = 0
        for r in range(N):
            for k in range(k_):
                s += int(x[r, o * Mb + i, k]) * int(w_kn[r, k, c])
        y[o, i, c] = s
    return y


@pytest.mark.parametrize("N,m,K,n", [(1, 3, 5, 4), (2, 4, 16, 3), (3, 2, 7, 5), (4, 8, 9, 2)])
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_ag_brute_force_exact(N, m, K, n, layout):
    x, w = gen.int_inputs((N, m, K), (N, K, n), -8, 8, seed=N * 100 + m)
    if layout == "nk":
        w = w.transpose(1, 2).contiguous()
    xb, wb = gen.bf16_bits(x), gen.bf16_bits(w)
    ref = _brute_ag(x.to(torch.int64).numpy(), _w_kn(w.to(torch.int64).numpy(), layout))
    got = oracle.ag_gemm(xb, wb, layout)
    assert np.array_equal(got, ref.astype(np.float64))


@pytest.mark.parametrize("N,Mb,k,n", [(1, 3, 5, 4), (2, 4, 16, 3), (3, 2, 7, 5), (4, 8, 9, 2)])
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_rs_brute_force_exact(N, Mb, k, n, layout):
    x, w = gen.int_inputs((N, N * Mb, k), (N, k, n), -8, 8, seed=N * 7 + k)
    if layout == "nk":
        w = w.transpose(1, 2).contiguous()
    ref = _brute_rs(x.to(torch.int64).numpy(), _w_kn(w.to(torch.int64).numpy(), layout))
    got = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), layout)
    assert np.array_equal(got, ref.astype(np.float64))


def test_sampled_rows_match_full():
    x, w = gen.ag_inputs(3, 16, 24, 10, gen.NORMAL1, gen.NORMAL002, seed=7, w_layout="kn")
    xb, wb = gen.bf16_bits(x), gen.bf16_bits(w)
    full = oracle.ag_gemm(xb, wb, "kn")
    ranks = np.array([0, 2, 1, 2, 0])
    rows = np.array([0, 47, 16, 15, 31])
    assert np.array_equal(oracle.ag_gemm_rows(xb, wb, ranks, rows, "kn"), full[ranks, rows])
    xr, wr = gen.rs_inputs(3, 12, 20, 9, gen.NORMAL1, gen.NORMAL002, seed=8, w_layout="nk")
    xrb, wrb = gen.bf16_bits(xr), gen.bf16_bits(wr)
    fr = oracle.gemm_rs(xrb, wrb, "nk")
    owners = np.array([2, 0, 1, 1])
    rws = np.array([3, 0, 2, 1])
    assert np.array_equal(oracle.gemm_rs_rows(xrb, wrb, owners, rws, "nk"), fr[owners, rws])


def test_closed_form_constant_inputs():
    # X = 1, W = 1: every AG output is K; every RS output is N*k.
    N, m, K, n = 3, 4, 40, 6
    x = torch.ones(N, m, K, dtype=torch.bfloat16)
    w = torch.ones(N, n, K, dtype=torch.bfloat16)
    assert np.all(oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk") == K)
    xr = torch.ones(N, N * m, K, dtype=torch.bfloat16)
    assert np.all(oracle.gemm_rs(gen.bf16_bits(xr), gen.bf16_bits(w), "nk") == N * K)


def test_closed_form_shard_scaled():
    # X_j = (j+1) * ones: the rows of shard j in Y_r are (j+1) * colsum(W_r).
    N, m, K, n = 4, 3, 8, 5
    x = torch.stack([torch.full((m, K), float(j + 1)) for j in range(N)]).to(torch.bfloat16)
    _, w = gen.int_inputs((1,), (N, K, n), -4, 4, seed=3)
    y = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "kn")
    colsum = w.to(torch.float64).sum(dim=1).numpy()      # [N][n]
    for r in range(N):
        for j in range(N):
            assert np.array_equal(y[r, j * m:(j + 1) * m], np.tile((j + 1) * colsum[r], (m, 1)))


@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_tagged_placement(layout):
    N, m, K, n = 4, 300, 16, 6
    x, w = gen.tagged_ag_inputs(N, m, K, n, layout)
    y = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), layout)
    for r in range(N):
        for j in range(N):
            rows = y[r, j * m:(j + 1) * m]
            for c in range(n):
                if (c + r) % 2 == 0:
                    assert np.all(rows[:, c] == j + 1)
                else:
                    assert np.array_equal(rows[:, c], np.arange(m) % 256)


def test_n1_is_plain_gemm():
    x, w = gen.ag_inputs(1, 37, 50, 23, gen.NORMAL1, gen.NORMAL002, seed=11, w_layout="kn")
    y = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "kn")[0]
    ref = _f64(x[0]) @ _f64(w[0])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    xr, wr = gen.rs_inputs(1, 29, 44, 17, gen.NORMAL1, gen.NORMAL002, seed=12, w_layout="kn")
    yr = oracle.gemm_rs(gen.bf16_bits(xr), gen.bf16_bits(wr), "kn")[0]
    np.testing.assert_allclose(yr, _f64(xr[0]) @ _f64(wr[0]), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("N", [2, 3, 5])
def test_allreduce_is_rs_then_ag(N):
    Mb, k, n = 6, 12, 7
    x, w = gen.rs_inputs(N, N * Mb, k, n, gen.NORMAL1, gen.NORMAL002, seed=20 + N, w_layout="kn")
    y = oracle.gemm_rs(gen.bf16_bits(x), gen.bf16_bits(w), "kn")
    gathered = np.concatenate([y[o] for o in range(N)], axis=0)       # AllGather of the buckets
    x_cat = np.concatenate([_f64(x[r]) for r in range(N)], axis=1)    # [M][N*k]
    w_cat = np.concatenate([_f64(w[r]) for r in range(N)], axis=0)    # [N*k][n]
    np.testing.assert_allclose(gathered, x_cat @ w_cat, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
@pytest.mark.parametrize("chunks", [1, 2, 4])
def test_ag_ring_equals_definition_bitwise(N, direction, chunks):
    m, K, n = 8, 24, 5
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=30 + N, w_layout="nk")
    xb, wb = gen.bf16_bits(x), gen.bf16_bits(w)
    ref = oracle.ag_gemm(xb, wb, "nk")
    got = ring.ag_gemm_ring(xb, wb, "nk", chunks=chunks, direction=direction)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
@pytest.mark.parametrize("chunks", [1, 2])
def test_rs_ring_equals_definition(N, direction, chunks):
    Mb, k, n = 4, 16, 6
    x, w = gen.rs_inputs(N, N * Mb, k, n, gen.NORMAL1, gen.NORMAL002, seed=40 + N, w_layout="kn")
    xb, wb = gen.bf16_bits(x), gen.bf16_bits(w)
    ref = oracle.gemm_rs(xb, wb, "kn")
    got = ring.gemm_rs_ring(xb, wb, "kn", chunks=chunks, direction=direction)
    assert not np.isnan(got).any()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("N", [2, 3, 4, 7, 8])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
def test_ag_ring_schedule_properties(N, direction):
    """Every rank uses every shard once; a shard reaches rank r at step i only
    from the neighbour that held it at step i-1 (so step i uses only shards
    already resident)."""
    m, K, n = 4, 8, 3
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=1, w_layout="nk")
    _, log = ring.ag_gemm_ring(gen.bf16_bits(x), gen.bf16_bits(w), "nk",
                               direction=direction, return_log=True)
    got = {r: {r} for r in range(N)}
    for step, stream, src, dst, obj, chunk in log:
        step_sign = 1 if stream == "cw" else -1
        assert dst == (src + step_sign) % N
        # the sender held that shard: either its own (step 0) or it arrived one hop earlier
        if step == 0:
            assert obj == src
        else:
            assert (src - step_sign * step) % N == obj
        got[dst].add(obj)
    for r in range(N):
        assert got[r] == set(range(N))
    assert len(log) == N * (N - 1)    # each rank receives each foreign shard exactly once


@pytest.mark.parametrize("N", [2, 3, 4, 7, 8])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
def test_rs_ring_bucket_visits(N, direction):
    """Each bucket visits every non-owner rank exactly once and ends on its owner."""
    Mb, k, n = 2, 4, 3
    x, w = gen.rs_inputs(N, N * Mb, k, n, gen.NORMAL1, gen.NORMAL002, seed=2, w_layout="nk")
    _, log = ring.gemm_rs_ring(gen.bf16_bits(x), gen.bf16_bits(w), "nk",
                               direction=direction, return_log=True)
    visits = {o: [] for o in range(N)}
    for step, stream, src, dst, obj, chunk in log:
        visits[obj].append(src)
    for o in range(N):
        assert sorted(visits[o]) == sorted(set(range(N)) - {o})
    if direction == "uni":
        assert len(log) == N * (N - 1)


def test_dropped_message_times_out():
    x, w = gen.ag_inputs(4, 4, 8, 3, gen.NORMAL1, gen.NORMAL002, seed=1, w_layout="nk")
    with pytest.raises(ring.RingTimeout, match="rank 2"):
        ring.ag_gemm_ring(gen.bf16_bits(x), gen.bf16_bits(w), "nk",
                          drop={(1, 0, "cw")}, timeout=0.5)
    xr, wr = gen.rs_inputs(3, 6, 4, 3, gen.NORMAL1, gen.NORMAL002, seed=1, w_layout="nk")
    with pytest.raises(ring.RingTimeout):
        ring.gemm_rs_ring(gen.bf16_bits(xr), gen.bf16_bits(wr), "nk",
                          drop={(0, 1, "cw")}, timeout=0.5)


# ---- planted mistakes: each must fail one of the pins above ----------------

def test_plant_transposed_operand_fails_brute_force():
    N, m, K, n = 2, 3, 6, 6     # square W so a transposed read is well-formed
    x, w = gen.int_inputs((N, m, K), (N, K, n), -8, 8, seed=5)
    ref = _brute_ag(x.to(torch.int64).numpy(), w.to(torch.int64).numpy())
    wrong = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")   # reads W^T
    assert not np.array_equal(wrong, ref.astype(np.float64))


def test_plant_shifted_placement_fails_tagged():
    N, m, K, n = 3, 5, 4, 4
    x, w = gen.tagged_ag_inputs(N, m, K, n, "nk")
    y = oracle.ag_gemm(gen.bf16_bits(x), gen.bf16_bits(w), "nk")
    shifted = np.roll(y, m, axis=1)           # shard j written into the rows of shard j+1
    assert not np.all(shifted[0, 0:m, 0] == 1)


def test_plant_dropped_contribution_fails_allreduce():
    N, Mb, k, n = 3, 4, 8, 5
    x, w = gen.rs_inputs(N, N * Mb, k, n, gen.NORMAL1, gen.NORMAL002, seed=9, w_layout="kn")
    x_drop = x.clone()
    x_drop[1] = 0                              # rank 1's contribution missing
    y = oracle.gemm_rs(gen.bf16_bits(x_drop), gen.bf16_bits(w), "kn")
    x_cat = np.concatenate([_f64(x[r]) for r in range(N)], axis=1)
    w_cat = np.concatenate([_f64(w[r]) for r in range(N)], axis=0)
    assert not np.allclose(np.concatenate(list(y), axis=0), x_cat @ w_cat, rtol=1e-6)


def test_plant_wrong_neighbour_fails_ring(monkeypatch):
    """A ring whose counter-clockwise stream goes the wrong way hands ranks
    shards they already used; the definition check must catch it."""
    N, m, K, n = 5, 4, 8, 3
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=4, w_layout="nk")
    xb, wb = gen.bf16_bits(x), gen.bf16_bits(w)
    ref = oracle.ag_gemm(xb, wb, "nk")
    real_send = ring._Net.send

    def bad_send(self, src, dst, stream, step, obj, chunk, payload):
        if stream == "ccw":
            dst = (src + 1) % self.N           # planted: wrong neighbour sign
        return real_send(self, src, dst, stream, step, obj, chunk, payload)

    monkeypatch.setattr(ring._Net, "send", bad_send)
    got = None
    try:
        got = ring.ag_gemm_ring(xb, wb, "nk", direction="bidi", timeout=0.5)
    except ring.RingTimeout:
        return                                  # caught: the schedule stalls
    assert not np.array_equal(got, ref)


# --- the backward pair of the column-parallel layer ("Tensor Parallelism >
# Communication Patterns": the backward pass is the forward's dual; "Hiding
# Tensor-Parallel Collectives", section 7: the weight gradient needs an
# AllGather of the input that the data gradient does not) -----------------

def _brute_wgrad(x, dy):
    """Pure-Python exact sums: dW_r[i][k] = sum_t dY_r[t][i] * X_all[t][k]."""
    N, m, K = x.shape
    n = dy.shape[2]
    x_all = x.reshape(N * m, K)
    out = np.zeros((N, n, K), dtype=np.int64)
    for r, i, k in itertools.product(range(N), range(n), range(K)):
        s = 0
        for t in range(N * m):
            s += int(dy[r, t, i]) * int(x_all[t, k])
        out[r, i, k] = s
    return out


@pytest.mark.parametrize("N,m,K,n", [(1, 3, 5, 4), (2, 4, 6, 3), (3, 2, 7, 5), (4, 3, 4, 2)])
def test_wgrad_brute_force_exact(N, m, K, n):
    x, _ = gen.int_inputs((N, m, K), (1, 1), -8, 8, seed=N * 31 + m)
    dy, _ = gen.int_inputs((N, N * m, n), (1, 1), -8, 8, seed=N * 37 + n)
    ref = _brute_wgrad(x.to(torch.int64).numpy(), dy.to(torch.int64).numpy())
    got = oracle.wgrad(gen.bf16_bits(x), gen.bf16_bits(dy))
    assert np.array_equal(got, ref.astype(np.float64))


def test_wgrad_all_ones_gradient_is_column_sums():
    N, m, K, n = 3, 5, 7, 4
    x, _ = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=8)
    dy = torch.ones((N, N * m, n), dtype=torch.bfloat16)
    got = oracle.wgrad(gen.bf16_bits(x), gen.bf16_bits(dy))
    colsum = _f64(x).reshape(N * m, K).sum(axis=0)
    assert np.allclose(got, np.broadcast_to(colsum, (N, n, K)), rtol=1e-13, atol=1e-12)


def test_wgrad_equals_numpy_transpose_matmul():
    N, m, K, n = 4, 6, 9, 5
    x, _ = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL002, seed=9)
    dy, _ = gen.ag_inputs(N, N * m, n, 1, gen.NORMAL1, gen.NORMAL002, seed=10)
    got = oracle.wgrad(gen.bf16_bits(x), gen.bf16_bits(dy))
    x_all = _f64(x).reshape(N * m, K)
    for r in range(N):
        assert np.allclose(got[r], _f64(dy)[r].T @ x_all, rtol=1e-12, atol=1e-12)
    rows = oracle.wgrad_rows(gen.bf16_bits(x), gen.bf16_bits(dy), [0, 3, 2], [4, 0, 2])
    assert np.array_equal(rows, got[[0, 3, 2], [4, 0, 2]])


@pytest.mark.parametrize("N", [1, 2, 4])
def test_backward_pair_adjoint_identities(N):
    """<dY, dL/dY-linear map> identities: for Y_r = X_all @ W_r^T,
    sum_r <dY_r, Y_r> = sum_r <dW_r, W_r> (wgrad) = sum_j <dX_j, X_j> (dgrad,
    the GEMM->ReduceScatter of dY_r @ W_r)."""
    m, K, n = 4, 6, 5
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL1, seed=20 + N, w_layout="nk")   # W_r [n][K]
    dy, _ = gen.ag_inputs(N, N * m, n, 1, gen.NORMAL1, gen.NORMAL1, seed=30 + N)
    xb, wb, dyb = gen.bf16_bits(x), gen.bf16_bits(w), gen.bf16_bits(dy)
    y = oracle.ag_gemm(xb, wb, "nk")                           # [N][N*m][n]
    lhs = float((_f64(dy) * y).sum())
    dw = oracle.wgrad(xb, dyb)                                  # [N][n][K]
    assert float((dw * _f64(w)).sum()) == pytest.approx(lhs, rel=1e-12, abs=1e-12)
    dx = oracle.gemm_rs(dyb, wb, "kn")                          # W_r [n][K] is [k][n_out]: dX [N][m][K]
    assert dx.shape == (N, m, K)
    assert float((dx * _f64(x)).sum()) == pytest.approx(lhs, rel=1e-12, abs=1e-12)


def test_plant_wgrad_wrong_token_order_fails_identity():
    """A gradient that pairs dY rows with the wrong token (shard order reversed)
    breaks the adjoint identity."""
    N, m, K, n = 3, 4, 5, 3
    x, w = gen.ag_inputs(N, m, K, n, gen.NORMAL1, gen.NORMAL1, seed=41, w_layout="nk")
    dy, _ = gen.ag_inputs(N, N * m, n, 1, gen.NORMAL1, gen.NORMAL1, seed=42)
    xb, wb, dyb = gen.bf16_bits(x), gen.bf16_bits(w), gen.bf16_bits(dy)
    lhs = float((_f64(dy) * oracle.ag_gemm(xb, wb, "nk")).sum())
    bad = oracle.wgrad(xb[::-1].copy(), dyb)                   # X_all built from reversed shards
    assert abs(float((bad * _f64(w)).sum()) - lhs) > 1e-6 * max(1.0, abs(lhs))


# --- Cannon-style 2-D rotation ("Overlap Communication with Dependent
# Computation via Decomposition ...", section "What people did before") ----

def _cannon_blocks(q, bm, bk, bn, seed, layout="nk"):
    a, _ = gen.ag_inputs(q * q, bm, bk, 1, gen.NORMAL1, gen.NORMAL002, seed=seed)
    bshape = (q * q, bn, bk) if layout == "nk" else (q * q, bk, bn)
    b, _ = gen.ag_inputs(bshape[0], bshape[1], bshape[2], 1, gen.NORMAL1, gen.NORMAL002, seed=seed + 1)
    return a, b


def _assemble(a, b, q, layout):
    """Plain matrices: A [q*bm][q*bk] and B as a [q*bk][q*bn] "kn" operand."""
    P, bm, bk = a.shape
    A = a.reshape(q, q, bm, bk).permute(0, 2, 1, 3).reshape(q * bm, q * bk)
    bb = b if layout == "kn" else b.transpose(1, 2)          # blocks as [bk][bn]
    bn = bb.shape[2]
    B = bb.reshape(q, q, bk, bn).permute(0, 2, 1, 3).reshape(q * bk, q * bn)
    return A.contiguous(), B.contiguous()


@pytest.mark.parametrize("q", [1, 2, 3, 4])
@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_cannon_ring_equals_definition(q, layout):
    bm, bk, bn = 5, 6, 4
    a, b = _cannon_blocks(q, bm, bk, bn, seed=50 + q, layout=layout)
    c = ring.cannon_gemm(gen.bf16_bits(a), gen.bf16_bits(b), q, layout)
    A, B = _assemble(a, b, q, layout)
    ref = oracle.gemm(gen.bf16_bits(A), gen.bf16_bits(B), "kn")      # [q*bm][q*bn]
    got = c.reshape(q, q, bm, bn).transpose(0, 2, 1, 3).reshape(q * bm, q * bn)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("q", [2, 3, 4])
def test_cannon_schedule_properties(q):
    """A moves only to the left neighbour, B only up; every rank holds every
    contraction block exactly once."""
    a, b = _cannon_blocks(q, 2, 3, 2, seed=60)
    _, log = ring.cannon_gemm(gen.bf16_bits(a), gen.bf16_bits(b), q, "nk", return_log=True)
    held = {rho: set() for rho in range(q * q)}
    for rho in range(q * q):
        i, j = divmod(rho, q)
        held[rho].add((i + j) % q)
    for step, stream, src, dst, obj, _ in log:
        si, sj = divmod(src, q)
        di, dj = divmod(dst, q)
        if stream == "a":
            assert (di, dj) == (si, (sj - 1) % q) and obj[0] == di
            held[dst].add(obj[1])
        else:
            assert (di, dj) == ((si - 1) % q, sj) and obj[1] == dj
    assert all(h == set(range(q)) for h in held.values())
    assert len(log) == 2 * q * q * (q - 1)


def test_cannon_dropped_message_times_out():
    a, b = _cannon_blocks(2, 2, 2, 2, seed=70)
    with pytest.raises(ring.RingTimeout):
        ring.cannon_gemm(gen.bf16_bits(a), gen.bf16_bits(b), 2, "nk", drop={(0, 0, "a")}, timeout=0.5)


def test_plant_cannon_without_skew_fails_definition(monkeypatch):
    """Starting every rank from k = 0 (no skew) pairs mismatched blocks."""
    q, bm, bk, bn = 3, 3, 4, 2
    a, b = _cannon_blocks(q, bm, bk, bn, seed=80)
    src = open(ring.__file__).read()
    assert "k0 = (i + j) % q" in src
    bad_ns = {"__name__": "oracle.ring", "__package__": "oracle"}
    exec(compile(src.replace("k0 = (i + j) % q", "k0 = 0").replace(
        'assert a_id[1] == b_id[0], "the held blocks share the contraction index"', "pass"),
        ring.__file__, "exec"), bad_ns)
    c = bad_ns["cannon_gemm"](gen.bf16_bits(a), gen.bf16_bits(b), q, "nk")
    A, B = _assemble(a, b, q, "nk")
    ref = oracle.gemm(gen.bf16_bits(A), gen.bf16_bits(B), "kn")
    got = c.reshape(q, q, bm, bn).transpose(0, 2, 1, 3).reshape(q * bm, q * bn)
    assert not np.allclose(got, ref, rtol=1e-6, atol=1e-6)
