"""The cost model that gates the decomposition ("Overlap Communication with
Dependent Computation via Decomposition in Large Deep Learning Models",
sections "The idea" -- knowing when to decline -- and "What it costs").

The model is an event simulation of one rank; these tests pin it to the
closed forms it must reduce to where the answer is known in closed form
(compute-bound and transfer-bound rings, chunked pipelines, the native
collective), to the decisions the pages describe (decline thin compute,
keep big compute decomposed, prefer the bidirectional ring when transfer
dominates), and to monotonicity in every rate."""

import itertools
import math
import random

import pytest

from collective_matmul_decomposition_gb300 import cm

AG, RS = cm.CM_OP_AG_GEMM, cm.CM_OP_GEMM_RS


@pytest.fixture(scope="module", autouse=True)
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return cm.load()


def rates(tflops=1000.0, ring=400.0, coll=800.0, hop=0.0, mem=4000.0):
    return dict(gemm_tflops=tflops, ring_gbs=ring, coll_gbs=coll, hop_us=hop, mem_gbs=mem)


def ag_parts(r, m, K, n, c=1):
    """Per-chunk GEMM and transfer times (us) of one AG shard."""
    t_c = 2.0 * m * K * n / (r["gemm_tflops"] * 1e6) / c
    t_x = m * K * 2.0 / (r["ring_gbs"] * 1e3) / c
    return t_c, t_x


def rs_parts(r, N, M, k, n, c=1):
    rows = M / N
    t_c = 2.0 * rows * k * n / (r["gemm_tflops"] * 1e6) / c
    t_x = rows * n * 4.0 / (r["ring_gbs"] * 1e3) / c
    return t_c, t_x


@pytest.mark.parametrize("N", [2, 3, 8, 16])
def test_ag_compute_bound_is_n_gemms(N):
    r = rates(ring=1e6)   # transfers far faster than compute
    m, K, n = 1024, 8192, 3584
    t_c, t_x = ag_parts(r, m, K, n)
    assert t_x < t_c
    assert cm.cost_estimate(N, 1, "uni", AG, m, K, n, r) == pytest.approx(N * t_c, rel=1e-12)


@pytest.mark.parametrize("N", [2, 4, 8])
@pytest.mark.parametrize("c", [1, 2, 4])
def test_ag_transfer_bound_pipeline(N, c):
    """Links busy back to back: (N-1) shard transfers, then the last chunk's GEMM."""
    r = rates(tflops=1e6, ring=10.0)
    m, K, n = 512, 4096, 256
    t_c, t_x = ag_parts(r, m, K, n)
    assert t_c < t_x
    want = (N - 1) * t_x + t_c / c
    assert cm.cost_estimate(N, c, "uni", AG, m, K, n, r) == pytest.approx(want, rel=1e-12)


@pytest.mark.parametrize("N", [2, 5, 8])
def test_ag_hop_latency_adds_per_hop(N):
    r = rates(tflops=1e6, ring=10.0, hop=7.0)
    m, K, n = 512, 4096, 256
    t_c, t_x = ag_parts(r, m, K, n)
    want = (N - 1) * (t_x + 7.0) + t_c
    assert cm.cost_estimate(N, 1, "uni", AG, m, K, n, r) == pytest.approx(want, rel=1e-12)


@pytest.mark.parametrize("N", [4, 8, 16])
def test_ag_bidi_transfer_bound_halves_the_trips(N):
    """Even N: N/2 clockwise hops carry the farthest shard; ccw runs alongside."""
    r = rates(tflops=1e6, ring=10.0)
    m, K, n = 512, 4096, 256
    t_c, t_x = ag_parts(r, m, K, n)
    assert 2 * t_c < t_x
    want = (N // 2) * t_x + t_c   # the last step multiplies one shard
    assert cm.cost_estimate(N, 1, "bidi", AG, m, K, n, r) == pytest.approx(want, rel=1e-12)


@pytest.mark.parametrize("N", [2, 8, 16])
def test_rs_compute_bound(N):
    r = rates(ring=1e6)
    M, k, n = 8192, 3584, 8192
    t_c, t_x = rs_parts(r, N, M, k, n)
    assert t_x < t_c
    assert cm.cost_estimate(N, 1, "uni", RS, M, k, n, r) == pytest.approx(N * t_c, rel=1e-12)


@pytest.mark.parametrize("N", [2, 4, 8])
@pytest.mark.parametrize("c", [1, 2, 4])
def test_rs_transfer_bound_pipeline(N, c):
    """The first chunk's product, then (N-1) bucket transfers back to back."""
    r = rates(tflops=1e6, ring=10.0)
    M, k, n = 4096, 256, 4096
    t_c, t_x = rs_parts(r, N, M, k, n)
    assert t_c < t_x
    want = t_c / c + (N - 1) * t_x
    assert cm.cost_estimate(N, c, "uni", RS, M, k, n, r) == pytest.approx(want, rel=1e-12)


def test_native_is_collective_then_gemm():
    r = rates()
    N, m, K, n = 8, 512, 4096, 2048
    want = (N - 1) * m * K * 2 / (r["coll_gbs"] * 1e3) + 2.0 * N * m * K * n / (r["gemm_tflops"] * 1e6)
    assert cm.cost_estimate(N, 1, "none", AG, m, K, n, r) == pytest.approx(want, rel=1e-12)
    M, k = 4096, 256
    want = 2.0 * M * k * n / (r["gemm_tflops"] * 1e6) + (N - 1) * (M / N) * n * 4 / (r["coll_gbs"] * 1e3)
    assert cm.cost_estimate(N, 1, "none", RS, M, k, n, r) == pytest.approx(want, rel=1e-12)
    # one rank: nothing to move, every direction is the plain GEMM
    for d in ("uni", "bidi", "none"):
        assert cm.cost_estimate(1, 1, d, AG, m, K, n, r) == pytest.approx(2.0 * m * K * n / 1e9, rel=1e-12)


def test_declines_thin_compute():
    """A thin GEMM-RS (k = 256 per rank, fp32 buckets) cannot hide the ring's
    slower transfer: keep the native collective."""
    r = rates(tflops=1000.0, ring=100.0, coll=600.0)
    t_c, t_x = rs_parts(r, 8, 4096, 256, 4096)
    assert t_c < t_x / 10
    c, d, us = cm.plan_choose(8, RS, 4096, 256, 4096, r)
    assert d == "none" and c == 1
    assert us == pytest.approx(cm.cost_estimate(8, 1, "none", RS, 4096, 256, 4096, r))


def test_keeps_big_compute_decomposed():
    r = rates(tflops=1000.0, ring=600.0, coll=900.0)
    t_c, t_x = ag_parts(r, 1024, 8192, 3584)
    assert t_x < t_c
    c, d, us = cm.plan_choose(8, AG, 1024, 8192, 3584, r)
    assert d == "uni" and c == 1   # compute hides every transfer; ties keep the simplest ring
    assert us < cm.cost_estimate(8, 1, "none", AG, 1024, 8192, 3584, r)


def test_prefers_bidi_when_transfer_dominates():
    r = rates(tflops=1000.0, ring=50.0, coll=60.0)
    c, d, _ = cm.plan_choose(8, AG, 2048, 4096, 512, r)
    assert d == "bidi"


def test_more_chunks_only_when_they_pay():
    """Chunks shorten the exposed first transfer; with hop latency they cost."""
    base = rates(tflops=1000.0, ring=100.0, coll=150.0)
    N, m, K, n = 8, 4096, 4096, 1024
    no_lat = [cm.cost_estimate(N, c, "uni", AG, m, K, n, base) for c in (1, 2, 4, 8)]
    assert no_lat == sorted(no_lat, reverse=True)
    slow = dict(base, hop_us=500.0)
    lat = [cm.cost_estimate(N, c, "uni", AG, m, K, n, slow) for c in (1, 2, 4, 8)]
    assert lat[0] < lat[-1]


def test_choice_is_the_minimum_over_candidates():
    rnd = random.Random(5)
    for _ in range(40):
        r = rates(tflops=rnd.uniform(50, 2000), ring=rnd.uniform(5, 900), coll=rnd.uniform(5, 900),
                  hop=rnd.uniform(0, 50), mem=rnd.uniform(500, 8000))
        N = rnd.choice([2, 3, 4, 8, 16])
        op = rnd.choice([AG, RS])
        rows = N * rnd.choice([64, 256, 1024]) if op == RS else rnd.choice([64, 256, 1024])
        K, n = rnd.choice([256, 4096]), rnd.choice([512, 8192])
        c, d, us = cm.plan_choose(N, op, rows, K, n, r)
        unit = rows if op == AG else rows // N
        cands = [cm.cost_estimate(N, 1, "none", op, rows, K, n, r)]
        cands += [cm.cost_estimate(N, cc, dd, op, rows, K, n, r)
                  for dd in ("uni", "bidi") for cc in (1, 2, 4, 8) if unit % cc == 0]
        assert us == pytest.approx(min(cands), rel=1e-8)
        assert us == pytest.approx(cm.cost_estimate(N, c, d, op, rows, K, n, r), rel=1e-12)


@pytest.mark.parametrize("op", [AG, RS])
def test_monotone_in_every_rate(op):
    rnd = random.Random(11 + op)
    for _ in range(20):
        base = rates(tflops=rnd.uniform(100, 2000), ring=rnd.uniform(10, 900), coll=rnd.uniform(10, 900),
                     hop=rnd.uniform(0, 20), mem=rnd.uniform(500, 8000))
        N, c = rnd.choice([2, 4, 8]), rnd.choice([1, 2, 4])
        rows = 1024 * N if op == RS else 1024
        for d, key in itertools.product(("uni", "bidi", "none"), ("gemm_tflops", "ring_gbs", "coll_gbs", "mem_gbs")):
            t0 = cm.cost_estimate(N, c, d, op, rows, 2048, 4096, base)
            t1 = cm.cost_estimate(N, c, d, op, rows, 2048, 4096, dict(base, **{key: base[key] * 2}))
            assert t1 <= t0 * (1 + 1e-12), (d, key)
        t0 = cm.cost_estimate(N, c, "uni", op, rows, 2048, 4096, base)
        t1 = cm.cost_estimate(N, c, "uni", op, rows, 2048, 4096, dict(base, hop_us=base["hop_us"] + 5))
        assert t1 >= t0


def test_lower_bounds():
    """Never faster than the rank's own compute, nor than the farthest shard's trip."""
    r = rates(tflops=800.0, ring=200.0)
    for N, c, d in itertools.product((2, 4, 8), (1, 2, 4), ("uni", "bidi")):
        m, K, n = 1024, 4096, 2048
        t_c, t_x = ag_parts(r, m, K, n)
        trips = N - 1 if d == "uni" else N // 2
        t = cm.cost_estimate(N, c, d, AG, m, K, n, r)
        assert t >= N * t_c * (1 - 1e-12)
        assert t >= trips * t_x * (1 - 1e-12)


def test_argument_errors(lib):
    r = cm._rates(rates())
    us = __import__("ctypes").c_double()
    ref = __import__("ctypes").byref
    assert lib.cm_cost_estimate(0, 1, 0, AG, 64, 64, 64, ref(r), ref(us)) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_cost_estimate(4, 0, 0, AG, 64, 64, 64, ref(r), ref(us)) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_cost_estimate(4, 1, 7, AG, 64, 64, 64, ref(r), ref(us)) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_cost_estimate(4, 1, 0, 9, 64, 64, 64, ref(r), ref(us)) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_cost_estimate(4, 1, 0, RS, 66, 64, 64, ref(r), ref(us)) == cm.CM_ERR_SHAPE
    assert lib.cm_cost_estimate(4, 1, 0, AG, 64, 64, 64, None, ref(us)) == cm.CM_ERR_INVALID_ARG
    for bad in (dict(gemm_tflops=0.0), dict(ring_gbs=-1.0), dict(hop_us=-1.0), dict(mem_gbs=math.nan)):
        rb = cm._rates(dict(rates(), **bad))
        assert lib.cm_cost_estimate(4, 1, 0, AG, 64, 64, 64, ref(rb), ref(us)) == cm.CM_ERR_INVALID_ARG
    with pytest.raises(cm.CMError):
        cm.plan_choose(4, AG, 64, 64, 64, rates(), max_chunks=0)


# ---- one Einsum that offers both collectives ----------------------------------
# Per rank: gathered A [N*m, K] (N row shards [m, K]), weight [K, n], the
# [N*m, n] fp32 result summed over ranks and scattered in buckets of m rows.

def einsum_native(r, N, m, K, n):
    """Both collectives native around the GEMM (closed form)."""
    coll = r["coll_gbs"] * 1e3
    return ((N - 1) * m * K * 2 / coll + 2.0 * N * m * K * n / (r["gemm_tflops"] * 1e6)
            + (N - 1) * m * n * 4 / coll)


def test_einsum_native_closed_form():
    r = rates()
    for N, m, K, n in ((2, 64, 256, 512), (8, 512, 4096, 2048), (16, 128, 1024, 8192)):
        assert cm.einsum_cost(N, 1, "none", "none", m, K, n, r) == pytest.approx(einsum_native(r, N, m, K, n),
                                                                                  rel=1e-12)
        # a ring direction with nothing decomposed, or one rank, is the same thing
        assert cm.einsum_cost(N, 2, "uni", "none", m, K, n, r) == pytest.approx(einsum_native(r, N, m, K, n))
    assert cm.einsum_cost(1, 1, "uni", "ag", 64, 256, 512, r) == pytest.approx(einsum_native(r, 1, 64, 256, 512))


def test_einsum_each_decomposition_is_its_ring_plus_the_other_native():
    """Decomposing the gather = the AG ring (cm_cost_estimate) + native
    scatter; decomposing the scatter = native gather + the RS ring over the
    N*m gathered rows."""
    r = rates(tflops=700.0, ring=300.0, coll=500.0, hop=3.0)
    N, m, K, n = 8, 512, 4096, 2048
    coll = r["coll_gbs"] * 1e3
    for c, d in itertools.product((1, 2, 4), ("uni", "bidi")):
        want_ag = cm.cost_estimate(N, c, d, AG, m, K, n, r) + (N - 1) * m * n * 4 / coll
        want_rs = (N - 1) * m * K * 2 / coll + cm.cost_estimate(N, c, d, RS, N * m, K, n, r)
        assert cm.einsum_cost(N, c, d, "ag", m, K, n, r) == pytest.approx(want_ag, rel=1e-12)
        assert cm.einsum_cost(N, c, d, "rs", m, K, n, r) == pytest.approx(want_rs, rel=1e-12)


def test_einsum_free_communication_keeps_everything_native():
    """With free links nothing is gained by a ring: ties keep the native form."""
    r = rates(ring=1e12, coll=1e12, hop=0.0)
    w, c, d, us = cm.plan_choose_einsum(8, 512, 4096, 2048, r)
    assert (w, c, d) == ("none", 1, "none")
    assert us == pytest.approx(2.0 * 8 * 512 * 4096 * 2048 / (r["gemm_tflops"] * 1e6), rel=1e-9)


def test_einsum_decomposes_the_heavier_collective():
    """A wide contraction (K >> n) makes the gather the big transfer; a wide
    output (n >> K) makes the fp32 scatter the big one.  The choice follows."""
    r = rates(tflops=1000.0, ring=400.0, coll=500.0)
    w, _, _, _ = cm.plan_choose_einsum(8, 1024, 16384, 512, r)
    assert w == "ag"
    w, _, _, _ = cm.plan_choose_einsum(8, 1024, 512, 16384, r)
    assert w == "rs"


def test_einsum_declines_thin_compute():
    """Little compute and a slow ring: neither ring can hide its transfer."""
    r = rates(tflops=2000.0, ring=20.0, coll=600.0)
    w, c, d, us = cm.plan_choose_einsum(8, 256, 256, 256, r)
    assert (w, c, d) == ("none", 1, "none")
    assert us == pytest.approx(einsum_native(r, 8, 256, 256, 256), rel=1e-9)


def test_einsum_choice_is_the_minimum_over_candidates():
    rnd = random.Random(23)
    for _ in range(40):
        r = rates(tflops=rnd.uniform(50, 2000), ring=rnd.uniform(5, 900), coll=rnd.uniform(5, 900),
                  hop=rnd.uniform(0, 50), mem=rnd.uniform(500, 8000))
        N = rnd.choice([2, 3, 4, 8, 16])
        m, K, n = rnd.choice([64, 256, 1024]), rnd.choice([256, 4096]), rnd.choice([512, 8192])
        w, c, d, us = cm.plan_choose_einsum(N, m, K, n, r)
        cands = [cm.einsum_cost(N, 1, "none", "none", m, K, n, r)]
        cands += [cm.einsum_cost(N, cc, dd, ww, m, K, n, r)
                  for ww in ("ag", "rs") for dd in ("uni", "bidi") for cc in (1, 2, 4, 8) if m % cc == 0]
        assert us == pytest.approx(min(cands), rel=1e-8)
        assert us == pytest.approx(cm.einsum_cost(N, c, d, w, m, K, n, r), rel=1e-12)


def test_einsum_argument_errors(lib):
    ctypes = __import__("ctypes")
    r = cm._rates(rates())
    us = ctypes.c_double()
    assert lib.cm_einsum_cost(4, 1, 0, 5, 64, 64, 64, ctypes.byref(r), ctypes.byref(us)) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_einsum_cost(4, 1, 0, AG, 0, 64, 64, ctypes.byref(r), ctypes.byref(us)) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_einsum_cost(4, 1, 0, AG, 64, 64, 64, None, ctypes.byref(us)) == cm.CM_ERR_INVALID_ARG
    w, c, d = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert lib.cm_plan_choose_einsum(4, 64, 64, 64, ctypes.byref(r), 0, ctypes.byref(w), ctypes.byref(c),
                                     ctypes.byref(d), None) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_plan_choose_einsum(4, 64, 64, 64, ctypes.byref(r), 4, None, ctypes.byref(c),
                                     ctypes.byref(d), None) == cm.CM_ERR_INVALID_ARG
