"""Hand-worked examples (tests/golden/*.json) against the oracle and its ring simulation.

The pages print no numeric example, so each fixture is a tiny integer case
worked out by hand from the pages' description of the ring (cited in the
fixture): the result of every rank and the content of every message -- the
shard a rank forwards, or the partial bucket with the contributions added so
far.  Small integers are exact in bf16 and in fp64, so every comparison is
exact.  The CPU tests pin the oracle; the GPU test runs the same examples
through the C ABI, zero-padded to the TMA granule, and must reproduce them
bit for bit.
"""

import json
import os

import numpy as np
import pytest

import oracle
from oracle import ring

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def bits(values):
    """Small integers -> bf16 bit patterns (exact: the low 16 bits of the fp32 pattern are zero)."""
    f = np.asarray(values, dtype=np.float32)
    u = f.view(np.uint32)
    assert not (u & 0xFFFF).any(), "fixture values must be exact in bf16"
    return (u >> 16).astype(np.uint16)


def decoded(payload):
    p = np.asarray(payload)
    return oracle.bf16_to_f64(p) if p.dtype == np.uint16 else p.astype(np.float64)


def check_messages(trace, expected):
    got = sorted(((t[0], t[1], t[2], t[3], t[4]), decoded(t[6]).tolist()) for t in trace)
    want = sorted(((e["step"], e["stream"], e["src"], e["dst"], e["object"]),
                   np.asarray(e["payload"], dtype=np.float64).tolist()) for e in expected)
    assert got == want


def test_ag_worked_example_oracle():
    g = load("ag_gemm_n3_worked.json")
    y = oracle.ag_gemm(bits(g["x"]), bits(g["w"]), g["w_layout"])
    assert np.array_equal(y, np.asarray(g["y"], dtype=np.float64))


def test_ag_worked_example_ring_and_messages():
    g = load("ag_gemm_n3_worked.json")
    trace = []
    y = ring.ag_gemm_ring(bits(g["x"]), bits(g["w"]), g["w_layout"], trace=trace)
    assert np.array_equal(y, np.asarray(g["y"], dtype=np.float64))
    check_messages(trace, g["messages"])


def test_ag_worked_example_bidi_messages():
    """The bidirectional ring on the same three ranks: the own shard leaves
    both ways at step 0 and nothing is forwarded after it."""
    g = load("ag_gemm_n3_worked.json")
    trace = []
    y = ring.ag_gemm_ring(bits(g["x"]), bits(g["w"]), g["w_layout"], direction="bidi", trace=trace)
    assert np.array_equal(y, np.asarray(g["y"], dtype=np.float64))
    check_messages(trace, g["messages_bidi"])


def test_ag_worked_example_four_ranks_bidi():
    """Four ranks over the bidirectional ring: two clockwise hops (one
    forward at step 1) and one counter-clockwise hop, worked by hand; the
    oracle's definition and the ring give the same outputs."""
    g = load("ag_gemm_n4_bidi_worked.json")
    x, w = bits(g["x"]), bits(g["w"])
    want = np.asarray(g["y"], dtype=np.float64)
    assert np.array_equal(oracle.ag_gemm(x, w, g["w_layout"]), want)
    trace = []
    y = ring.ag_gemm_ring(x, w, g["w_layout"], direction="bidi", trace=trace)
    assert np.array_equal(y, want)
    check_messages(trace, g["messages_bidi"])
    # the one-way ring sends a different set of messages for the same result
    trace_uni = []
    ring.ag_gemm_ring(x, w, g["w_layout"], direction="uni", trace=trace_uni)
    with pytest.raises(AssertionError):
        check_messages(trace_uni, g["messages_bidi"])


def test_rs_worked_example_oracle():
    g = load("gemm_rs_n3_worked.json")
    y = oracle.gemm_rs(bits(g["x"]), bits(g["w"]), g["w_layout"])
    assert np.array_equal(y, np.asarray(g["y"], dtype=np.float64))


@pytest.mark.parametrize("direction", ["uni", "bidi"])
def test_rs_worked_example_ring_and_partial_buckets(direction):
    g = load("gemm_rs_n3_worked.json")
    trace = []
    y = ring.gemm_rs_ring(bits(g["x"]), bits(g["w"]), g["w_layout"], direction=direction, trace=trace)
    assert np.array_equal(y, np.asarray(g["y"], dtype=np.float64))
    check_messages(trace, g["messages_" + direction])


@pytest.mark.parametrize("direction", ["uni", "bidi"])
def test_rs_worked_example_four_ranks(direction):
    """Four ranks: three forwards per bucket one-way; two clockwise hops and
    one counter-clockwise hop on the bidirectional ring, whose owner adds
    partials of unequal length (the realigning addition)."""
    g = load("gemm_rs_n4_worked.json")
    x, w = bits(g["x"]), bits(g["w"])
    want = np.asarray(g["y"], dtype=np.float64)
    assert np.array_equal(oracle.gemm_rs(x, w, g["w_layout"]), want)
    trace = []
    y = ring.gemm_rs_ring(x, w, g["w_layout"], direction=direction, trace=trace)
    assert np.array_equal(y, want)
    check_messages(trace, g["messages_" + direction])


def test_plant_wrong_bucket_start_fails_worked_example():
    """A ring that started bucket o at rank o (instead of o+1) would still sum
    every contribution, but its messages would not be the hand-worked ones."""
    g = load("gemm_rs_n3_worked.json")
    x, w = bits(g["x"]), bits(g["w"])
    N = g["N"]
    shifted = [dict(e, src=(e["src"] - 1) % N, dst=(e["dst"] - 1) % N) for e in g["messages_uni"]]
    trace = []
    ring.gemm_rs_ring(x, w, g["w_layout"], trace=trace)
    with pytest.raises(AssertionError):
        check_messages(trace, shifted)


def test_cannon_worked_example():
    """Cannon's rotation on a 3 x 3 grid with 1 x 1 blocks: the product and
    the block every message carries (the skew, A moving left, B moving up),
    worked by hand; the oracle's definition agrees on the product."""
    g = load("cannon_q3_worked.json")
    q = g["q"]
    A = np.asarray(g["A"], dtype=np.float32)
    B = np.asarray(g["B"], dtype=np.float32)
    a_blocks = bits(A.reshape(q * q, 1, 1))                     # A_{i,k} at i*q + k
    b_blocks = bits(B.reshape(q * q, 1, 1))                     # B_{k,j} at k*q + j ("kn": [bk][bn])
    want = np.asarray(g["C"], dtype=np.float64).reshape(q * q, 1, 1)
    c, log = ring.cannon_gemm(a_blocks, b_blocks, q, g["b_layout"], return_log=True)
    assert np.array_equal(c, want)
    got = sorted((e[0], e[1], e[2], e[3], tuple(e[4])) for e in log)
    exp = sorted((m["step"], m["stream"], m["src"], m["dst"], tuple(m["block"])) for m in g["messages"])
    assert got == exp
    assert np.array_equal(oracle.gemm(bits(A), bits(B), "kn"), np.asarray(g["C"], dtype=np.float64))


@pytest.mark.gpu
@pytest.mark.parametrize("direction", ["uni", "bidi"])
def test_worked_examples_on_gpu(direction):
    """Both examples through the C ABI, K and n zero-padded to 8: the top-left
    block of every rank's output is the hand-worked result, exactly (fp32 out),
    and the padding stays zero."""
    import torch

    import __graft_entry__
    from collective_matmul_decomposition_gb300 import cm
    __graft_entry__.build()
    dev = "cuda:0"

    def pad(a, shape):
        t = torch.zeros(shape, dtype=torch.float32)
        a = torch.tensor(a, dtype=torch.float32)
        t[tuple(slice(0, s) for s in a.shape)] = a
        return t.to(torch.bfloat16).to(dev)

    g = load("ag_gemm_n3_worked.json")
    N, m = g["N"], len(g["x"][0])
    x = pad(g["x"], (N, m, 8))
    w = pad(g["w"], (N, 8, 8))             # [K][n] per rank
    plan = cm.Plan(N, 1, direction)
    ws = torch.full((plan.ag_workspace_size(m, 8),), 0xFF, dtype=torch.uint8, device=dev)
    y = torch.full((N, N * m, 8), float("nan"), dtype=torch.float32, device=dev)
    cm.cm_ag_gemm(plan, x, w, y, ws, "kn")
    assert cm.cm_check_status(ws)[0] == 0
    want = torch.zeros(N, N * m, 8, dtype=torch.float64)
    want[:, :, :2] = torch.tensor(g["y"], dtype=torch.float64)
    assert torch.equal(y.cpu().double(), want)

    g = load("gemm_rs_n3_worked.json")
    N, M = g["N"], len(g["x"][0])
    x = pad(g["x"], (N, M, 8))
    w = pad(g["w"], (N, 8, 8))
    ws = torch.full((plan.rs_workspace_size(M, 8),), 0xFF, dtype=torch.uint8, device=dev)
    y = torch.full((N, M // N, 8), float("nan"), dtype=torch.float32, device=dev)
    cm.cm_gemm_rs(plan, x, w, y, ws, "kn")
    assert cm.cm_check_status(ws)[0] == 0
    want = torch.zeros(N, M // N, 8, dtype=torch.float64)
    want[:, :, :2] = torch.tensor(g["y"], dtype=torch.float64)
    assert torch.equal(y.cpu().double(), want)
