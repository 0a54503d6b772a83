"""Rank-by-rank simulation of the ring schedules, in fp64 (test infrastructure).

Each logical rank runs as a thread that only talks to its two ring
neighbours through message queues, the way the pages describe the per-rank
loop; the schedule is derived here from the pages, independently of the
library's planner, and every message carries the id of the shard or bucket
it holds, so nothing in the arithmetic depends on an index formula.

* AllGather->GEMM ("Hiding Tensor-Parallel Collectives", section 3;
  "Overlap Communication ... via Decomposition", section "The idea"):
  a rank starts with its own shard, multiplies it while forwarding it to its
  neighbour, then multiplies what it received while forwarding that, until
  it has used all N shards; each partial product is written into the rows of
  its shard (DynamicUpdateSlice).
* GEMM->ReduceScatter (same pages, section 5 / "The idea"): an accumulating
  bucket circulates; a rank adds its contribution to the bucket it holds and
  forwards it; after visiting every rank the bucket rests at its owner.
* Bidirectional ring (section "The idea", bidirectional rings; section
  "What it costs", pre-shift and realigning addition): the N-1 foreign shards
  (AG) or contributions (RS) are split between a clockwise stream of
  a = ceil((N-1)/2) hops and a counter-clockwise stream of b = floor((N-1)/2)
  hops; in RS the owner adds the two partial buckets and its own contribution.
* Chunks ("Hiding Tensor-Parallel Collectives", sections 3 and 6): every
  shard / bucket travels as `chunks` contiguous row blocks, each a separate
  message; the result does not depend on the chunk count.

Ring direction reading: "clockwise" sends rank r -> r+1 (mod N).

A dropped message (fault injection) makes the receiving rank time out and
the simulation raise RingTimeout, naming the rank and step.
"""

from __future__ import annotations

import queue
import threading

import numpy as np

from . import gemm as _gemm


class RingTimeout(RuntimeError):
    pass


def hop_split(N: int):
    """(a, b): clockwise and counter-clockwise hop counts of the bidirectional ring."""
    a = (N - 1 + 1) // 2   # ceil((N-1)/2)
    b = (N - 1) // 2       # floor((N-1)/2)
    return a, b


class _Net:
    """Point-to-point links between neighbouring ranks, one inbox per (rank, stream)."""

    def __init__(self, N, streams, drop=None, timeout=5.0, trace=None):
        self.N = N
        self.boxes = {(r, s): queue.Queue() for r in range(N) for s in streams}
        self.drop = set(drop or ())   # {(sender, step, stream)}
        self.timeout = timeout
        self.log = []                 # (step, stream, src, dst, object id, chunk)
        self.trace = trace            # optional list: the log entries with a copy of each payload
        self.lock = threading.Lock()

    def send(self, src, dst, stream, step, obj, chunk, payload):
        with self.lock:
            self.log.append((step, stream, src, dst, obj, chunk))
            if self.trace is not None:
                self.trace.append((step, stream, src, dst, obj, chunk, np.array(payload, copy=True)))
        if (src, step, stream) in self.drop:
            return
        self.boxes[(dst, stream)].put((obj, chunk, payload))

    def recv(self, rank, stream, step):
        try:
            return self.boxes[(rank, stream)].get(timeout=self.timeout)
        except queue.Empty:
            raise RingTimeout(f"rank {rank} waited for step {step} ({stream}) "
                              f"longer than {self.timeout}s") from None


def _run(N, body):
    errors = []

    def wrap(r):
        try:
            body(r)
        except BaseException as e:  # noqa: BLE001 - reported to the caller
            errors.append(e)

    ts = [threading.Thread(target=wrap, args=(r,)) for r in range(N)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if errors:
        raise errors[0]


def _chunks(rows: int, chunks: int):
    assert rows % chunks == 0, "a shard splits into equal row chunks"
    h = rows // chunks
    return [(q * h, (q + 1) * h) for q in range(chunks)]


def ag_gemm_ring(x_bits, w_bits, w_layout="nk", chunks=1, direction="uni",
                 drop=None, timeout=5.0, return_log=False, trace=None):
    """AllGather->GEMM by the ring schedule; returns y [N][N*m][n] fp64."""
    x = np.ascontiguousarray(x_bits)
    w = np.ascontiguousarray(w_bits)
    N, m, K = x.shape
    n = w.shape[2] if w_layout == "kn" else w.shape[1]
    y = np.full((N, N * m, n), np.nan)
    spans = _chunks(m, chunks)
    if direction == "uni":
        hops = {"cw": N - 1}
    elif direction == "bidi":
        a, b = hop_split(N)
        hops = {"cw": a, "ccw": b}
    else:
        raise ValueError(direction)
    nxt = {"cw": lambda r: (r + 1) % N, "ccw": lambda r: (r - 1) % N}
    net = _Net(N, list(hops), drop, timeout, trace)

    def rank(r):
        # step 0: multiply the own shard, chunk by chunk, forwarding each chunk
        own = [(r, q, x[r, lo:hi]) for q, (lo, hi) in enumerate(spans)]
        for s, q, blk in own:
            lo, hi = spans[q]
            y[r, s * m + lo:s * m + hi] = _gemm(blk, w[r], w_layout)
            for st, h in hops.items():
                if h >= 1:
                    net.send(r, nxt[st](r), st, 0, s, q, blk)
        # later steps: use what arrived, forward it while hops remain
        for st, h in hops.items():
            for step in range(1, h + 1):
                for _ in spans:
                    s, q, blk = net.recv(r, st, step)
                    lo, hi = spans[q]
                    y[r, s * m + lo:s * m + hi] = _gemm(blk, w[r], w_layout)
                    if step < h:
                        net.send(r, nxt[st](r), st, step, s, q, blk)

    _run(N, rank)
    return (y, net.log) if return_log else y


def gemm_rs_ring(x_bits, w_bits, w_layout="nk", chunks=1, direction="uni",
                 drop=None, timeout=5.0, return_log=False, trace=None):
    """GEMM->ReduceScatter by the circulating-bucket schedule; y [N][M/N][n] fp64."""
    x = np.ascontiguousarray(x_bits)
    w = np.ascontiguousarray(w_bits)
    N, M, k = x.shape
    n = w.shape[2] if w_layout == "kn" else w.shape[1]
    Mb = M // N
    spans = _chunks(Mb, chunks)
    y = np.full((N, Mb, n), np.nan)
    nxt = {"cw": lambda r: (r + 1) % N, "ccw": lambda r: (r - 1) % N}

    def contrib(r, o, q):
        lo, hi = spans[q]
        return _gemm(x[r, o * Mb + lo:o * Mb + hi], w[r], w_layout)

    if direction == "uni":
        streams = ["cw"]
    elif direction == "bidi":
        streams = ["cw", "ccw"]
    else:
        raise ValueError(direction)
    net = _Net(N, streams, drop, timeout, trace)

    if direction == "uni":
        def rank(r):
            # a rank starts the bucket of its counter-clockwise neighbour, so
            # that after visiting all N ranks the bucket ends on its owner.
            o = (r - 1) % N
            for q in range(chunks):
                acc = contrib(r, o, q)
                if N == 1:
                    y[o, spans[q][0]:spans[q][1]] = acc
                else:
                    net.send(r, nxt["cw"](r), "cw", 0, o, q, acc)
            for step in range(1, N):
                for _ in range(chunks):
                    o, q, acc = net.recv(r, "cw", step)
                    acc = acc + contrib(r, o, q)
                    if o == r:                       # home: fully reduced
                        y[o, spans[q][0]:spans[q][1]] = acc
                    else:
                        net.send(r, nxt["cw"](r), "cw", step, o, q, acc)
    else:
        a, b = hop_split(N)

        def rank(r):
            partial = {}   # (stream, chunk) -> partial bucket that arrived home
            # clockwise: start the bucket owned by rank r+a; counter-clockwise:
            # start the bucket owned by rank r-b.
            starts = [("cw", a, (r + a) % N), ("ccw", b, (r - b) % N)]
            for st, h, o in starts:
                if h == 0:
                    continue
                for q in range(chunks):
                    acc = contrib(r, o, q)
                    dst = nxt[st](r)
                    net.send(r, dst, st, 0, o, q, acc)
            for st, h, _ in starts:
                for step in range(1, h + 1):
                    for _ in range(chunks):
                        o, q, acc = net.recv(r, st, step)
                        if o == r:                   # arrived home after h hops
                            partial[(st, q)] = acc
                        else:
                            acc = acc + contrib(r, o, q)
                            net.send(r, nxt[st](r), st, step, o, q, acc)
            # realigning addition at the owner: own contribution + both streams
            for q in range(chunks):
                tot = contrib(r, r, q)
                for st, h, _ in starts:
                    if h > 0:
                        tot = tot + partial[(st, q)]
                y[r, spans[q][0]:spans[q][1]] = tot

    _run(N, rank)
    return (y, net.log) if return_log else y


def cannon_gemm(a_bits, b_bits, q, b_layout="nk", drop=None, timeout=5.0, return_log=False):
    """Cannon-style 2-D rotation ("Overlap Communication with Dependent
    Computation via Decomposition ...", section "What people did before":
    shard rotation interleaved with partial products, operands split along
    the contracting dimension) on a q x q grid of ranks.

    a_bits: [q*q][bm][bk], block A_{i,k} at index i*q + k.
    b_bits: [q*q] blocks of B, B_{k,j} at index k*q + j, each [bn][bk]
            ("nk") or [bk][bn] ("kn").
    Rank (i, j) starts with A_{i,(i+j) mod q} and B_{(i+j) mod q, j} (the
    skew: with every block in one memory the rank simply starts from those),
    then for q steps multiplies what it holds into C_{i,j}, sends its A block
    to the left neighbour (i, j-1) and its B block to the upper neighbour
    (i-1, j), and receives the next ones from the right and from below.
    Returns C [q*q][bm][bn] fp64, C_{i,j} at index i*q + j.
    """
    a = np.ascontiguousarray(a_bits)
    b = np.ascontiguousarray(b_bits)
    P = q * q
    assert a.shape[0] == P and b.shape[0] == P
    bm = a.shape[1]
    bn = b.shape[1] if b_layout == "nk" else b.shape[2]
    c = np.full((P, bm, bn), np.nan)
    net = _Net(P, ["a", "b"], drop, timeout)

    def rank(rho):
        i, j = divmod(rho, q)
        k0 = (i + j) % q
        a_id, a_blk = (i, k0), a[i * q + k0]
        b_id, b_blk = (k0, j), b[k0 * q + j]
        acc = np.zeros((bm, bn))
        for s in range(q):
            assert a_id[1] == b_id[0], "the held blocks share the contraction index"
            acc += _gemm(a_blk, b_blk, b_layout)
            if s + 1 < q:
                net.send(rho, i * q + (j - 1) % q, "a", s, a_id, 0, a_blk)
                net.send(rho, ((i - 1) % q) * q + j, "b", s, b_id, 0, b_blk)
                a_id, _, a_blk = net.recv(rho, "a", s + 1)
                b_id, _, b_blk = net.recv(rho, "b", s + 1)
        c[rho] = acc

    _run(P, rank)
    return (c, net.log) if return_log else c
