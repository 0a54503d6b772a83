"""Host-side checks of the ring schedules and of the kernel's task table.

* cm_plan_step matches the schedule of the oracle's rank-by-rank ring
  simulation, which derives its own schedule from the pages.
* every flag a task waits on is signalled only by tasks of earlier steps, by
  exactly one task, so the kernel's static tile order cannot deadlock.
* an event-level simulation runs the task table the way the kernel does --
  G co-resident CTAs, each walking its tiles in order, flags as counters,
  slots / accumulator buffers as tagged contents -- under random interleaving
  and checks that every tile reads the shard or partial bucket it should and
  that every output ends with each rank's contribution exactly once.
"""

import random

import pytest

import __graft_entry__
from collective_matmul_decomposition_gb300 import cm
from collective_matmul_decomposition_gb300 import inputs as gen
from oracle import ring

AG, RS = cm.CM_OP_AG_GEMM, cm.CM_OP_GEMM_RS


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _plan_sends(p, op):
    out = set()
    streams = 2 if p.direction == "bidi" else 1
    for r in range(p.N):
        for i in range(p.steps(op)):
            for d in range(streams):
                obj, src, dst = p.step(op, r, i, d)
                if obj >= 0 and dst >= 0:
                    out.add((i, "cw" if d == 0 else "ccw", r, dst, obj))
    return out


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 13, 16])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
def test_schedule_matches_oracle_ring(N, direction):
    p = cm.Plan(N, 1, direction)
    x, w = gen.ag_inputs(N, 2, 8, 2, gen.NORMAL1, gen.NORMAL002, seed=1, w_layout="nk")
    _, log = ring.ag_gemm_ring(gen.bf16_bits(x), gen.bf16_bits(w), "nk", direction=direction,
                               return_log=True)
    assert _plan_sends(p, AG) == {(s, st, a, b, o) for (s, st, a, b, o, q) in log}
    xr, wr = gen.rs_inputs(N, 2 * N, 8, 2, gen.NORMAL1, gen.NORMAL002, seed=1, w_layout="nk")
    _, log = ring.gemm_rs_ring(gen.bf16_bits(xr), gen.bf16_bits(wr), "nk", direction=direction,
                               return_log=True)
    assert _plan_sends(p, RS) == {(s, st, a, b, o) for (s, st, a, b, o, q) in log}


@pytest.mark.parametrize("N", [1, 2, 3, 4, 7, 8, 16])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
def test_each_rank_uses_each_shard_once(N, direction):
    p = cm.Plan(N, 1, direction)
    for op in (AG, RS):
        tasks = p.tasks(op)
        assert len(tasks) == N * N
        pairs = sorted((t.rank, t.out_idx) for t in tasks)
        assert pairs == sorted((r, s) for r in range(N) for s in range(N))


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("direction", ["uni", "bidi", "none"])
@pytest.mark.parametrize("serial", [False, True])
@pytest.mark.parametrize("order", [0, 2])
@pytest.mark.parametrize("in_place", [2, 0])
def test_waits_point_to_earlier_tasks(N, direction, serial, order, in_place):
    """Every flag has exactly one signalling task, earlier in the table than
    every task waiting on it, and of an earlier ring step -- in the ring's
    own order (rank-blocked one-way, stream-blocked two-way) and in
    step-major order, for the GEMM-RS table of buckets in place and that of
    per-step buffers."""
    p = cm.Plan(N, 2, direction)
    p.set_option(cm.CM_OPT_RS_IN_PLACE, in_place)
    if serial:
        p.set_option(cm.CM_OPT_SERIAL_STEPS, 1)
    p.set_option(cm.CM_OPT_TASK_ORDER, order)
    for op in (AG, RS):
        tasks = p.tasks(op)
        if serial or direction == "none" or order == 2:
            assert [t.step for t in tasks] == sorted(t.step for t in tasks)
        signallers = {}
        for idx, t in enumerate(tasks):
            sigs = [t.sig_done] + ([t.sig_fwd[0], t.sig_fwd[1]] if op == AG else [])
            for s_ in sigs:
                if s_ >= 0:
                    assert s_ not in signallers, "a flag has one signaller"
                    signallers[s_] = (idx, t.step)
        for idx, t in enumerate(tasks):
            for f in list(t.wait_in) + list(t.wait_free):
                if f >= 0:
                    assert f in signallers, (op, f)
                    assert signallers[f][0] < idx
                    assert signallers[f][1] < t.step


@pytest.mark.parametrize("N", [3, 4, 8, 16])
def test_bidi_stream_blocked_runs(N):
    """A two-way ring's own order: clockwise tasks before counter-clockwise
    ones (owners aside), and each rank's tasks in at most five runs -- its
    weight shard is read that many times instead of once per step."""
    p = cm.Plan(N, 1, "bidi")
    for op in (AG, RS):
        tasks = p.tasks(op)
        streams = [t.stream for t in tasks if not (op == RS and t.out_buf < 0)]
        assert streams == sorted(streams)
        runs = {}
        prev = None
        for t in tasks:
            if t.rank != prev:
                runs[t.rank] = runs.get(t.rank, 0) + 1
            prev = t.rank
        assert max(runs.values()) <= 5, runs
        if N >= 8:
            assert max(runs.values()) < p.steps(op)


def test_step_major_order_is_a_permutation_of_the_ring_order():
    """CM_OPT_TASK_ORDER = 2 lists the same tasks, sorted by step then rank."""
    for d in ("uni", "bidi"):
        p = cm.Plan(8, 2, d)
        for op in (AG, RS):
            ring_order = p.tasks(op)
            p.set_option(cm.CM_OPT_TASK_ORDER, 2)
            sm = p.tasks(op)
            p.set_option(cm.CM_OPT_TASK_ORDER, 0)
            key = lambda t: (t.rank, t.step, t.stream, t.out_idx)
            assert sorted(map(key, ring_order)) == sorted(map(key, sm))
            assert [(t.step, t.rank) for t in sm] == sorted((t.step, t.rank) for t in sm)
    with pytest.raises(cm.CMError):
        cm.Plan(4, 1, "uni").set_option(cm.CM_OPT_TASK_ORDER, 3)


@pytest.mark.parametrize("N", [2, 3, 5, 8, 16])
def test_uni_ring_runs_each_rank_in_two_blocks(N):
    """One-way ring: each rank's tasks form at most two contiguous runs, in
    step order (so its weight shard streams twice, not once per step)."""
    p = cm.Plan(N, 1, "uni")
    for op in (AG, RS):
        ranks = [t.rank for t in p.tasks(op)]
        runs = {}
        prev = None
        for r in ranks:
            if r != prev:
                runs[r] = runs.get(r, 0) + 1
            prev = r
        assert max(runs.values()) <= 2
        for r in range(N):
            steps = [t.step for t in p.tasks(op) if t.rank == r]
            assert steps == sorted(steps) == list(range(N))


@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_tile_groups(group):
    """Groups are runs of at most `group` consecutive tasks of one rank."""
    p = cm.Plan(8, 2, "uni")
    p.set_option(cm.CM_OPT_TILE_GROUP, group)
    for op in (AG, RS):
        tasks = p.tasks(op)
        order = kernel_tile_order(tasks, 2, 3, 4)
        assert len(order) == len(tasks) * 2 * 3 * 4
        assert len(set(order)) == len(order)
        assert max(t.tile_group >> 8 for t in tasks) <= group
    for N in (2, 4):
        for d in ("uni", "bidi", "none"):
            q = cm.Plan(N, 1, d)
            q.set_option(cm.CM_OPT_TILE_GROUP, group)
            q.set_option(cm.CM_OPT_SERIAL_STEPS, 1)
            assert all(t.tile_group >> 8 == 1 for t in q.tasks(AG) + q.tasks(RS))


def test_slots_written_once():
    """Every receive slot (AG) has one writer; so does every RS accumulator
    buffer when buckets live in per-step buffers."""
    for d in ("uni", "bidi"):
        p = cm.Plan(8, 1, d)
        ag = [s_ for t in p.tasks(AG) for s_ in t.fwd_slot if s_ >= 0]
        assert len(ag) == len(set(ag))
        p.set_option(cm.CM_OPT_RS_IN_PLACE, 0)
        rs = [t.out_buf for t in p.tasks(RS) if t.out_buf >= 0]
        assert len(rs) == len(set(rs))
        assert all(t.in_buf[0] != t.out_buf or t.out_buf < 0 for t in p.tasks(RS))


@pytest.mark.parametrize("N", [2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
def test_in_place_buckets_form_one_chain_each(N, direction):
    """Buckets accumulated in place: each (bucket, stream) buffer is started by
    one task (no input), then updated in place (in_buf[0] == out_buf) by one
    task per later ring step, each waiting on its predecessor's flag, and read
    by the owner last -- a chain along the ring, one rank at a time."""
    p = cm.Plan(N, 1, direction)
    tasks = p.tasks(RS)
    streams = 2 if direction == "bidi" else 1
    users = {}
    for t in tasks:
        if t.out_buf >= 0:
            assert t.in_buf[1] < 0
            assert t.in_buf[0] in (-1, t.out_buf)
            assert t.out_buf // streams == t.out_idx and t.out_buf % streams == t.stream
            users.setdefault(t.out_buf, []).append(t)
        else:
            for j in range(2):
                if t.in_buf[j] >= 0:
                    assert t.in_buf[j] // streams == t.out_idx == t.rank
                    users.setdefault(t.in_buf[j], []).append(t)
    bufs_per_stream = set(b for b in users)
    assert len(bufs_per_stream) <= N * streams
    sig_of = {t.sig_done: t for t in tasks if t.sig_done >= 0}
    for b, ts in users.items():
        chain = sorted(ts, key=lambda t: t.step)
        # contributors at steps 0, 1, ...; the owner (step a of a two-way ring) last
        assert [t.step for t in chain[:-1]] == list(range(len(chain) - 1))
        assert chain[-1].step > chain[-2].step if len(chain) > 1 else True
        assert chain[0].in_buf[0] == -1 and chain[0].wait_in[0] < 0 and chain[0].out_buf == b
        for prev, cur in zip(chain, chain[1:]):
            j = 0 if cur.out_buf >= 0 or cur.in_buf[0] == b else 1
            assert cur.wait_in[j] == prev.sig_done and sig_of[prev.sig_done] is prev
        ranks = [t.rank for t in chain]
        assert len(set(ranks)) == len(ranks)
        assert chain[-1].out_buf < 0 and chain[-1].rank == b // streams   # the owner reads it last


def kernel_tile_order(tasks, c, mtiles, ntiles, band=0, slabs=1):
    """The kernels' tile order: with column slabs (GEMM-RS), one pass over
    the whole order per slab of ntiles / slabs column tiles; in a pass, task
    groups (cm_task.tile_group) in table order; inside a group chunk, row
    band (`band` row tiles of the group's task-by-task row tiles; 0 = one
    band), column tile, row tile of the band."""
    assert ntiles % slabs == 0
    nts = ntiles // slabs
    out = []
    for slab in range(slabs):
        t = 0
        while t < len(tasks):
            size = tasks[t].tile_group >> 8
            assert size >= 1 and all((tasks[t + j].tile_group & 0xff) == j for j in range(size))
            assert len({tasks[t + j].rank for j in range(size)}) == 1, "a group is one rank's tasks"
            rows = size * mtiles
            b = band if 0 < band < rows else rows
            for q in range(c):
                for b0 in range(0, rows, b):
                    for g in range(nts):
                        for rho in range(b0, min(rows, b0 + b)):
                            out.append((t + rho // mtiles, q, rho % mtiles, slab * nts + g))
            t += size
    return out


def _simulate(p, op, mtiles, ntiles, grid, seed, band=0, slabs=1):
    """Run the task table like the kernel: returns final outputs (see module doc)."""
    rnd = random.Random(seed)
    N, c = p.N, p.chunks
    tasks = p.tasks(op)
    tiles = kernel_tile_order(tasks, c, mtiles, ntiles, band, slabs)
    # readiness counters as the kernels keep them: AG one per (flag, chunk,
    # row tile) -- the row tile's forward (column tile 0 here, as the
    # single-CTA kernel does) bumps it once; RS one per (flag, chunk, row
    # tile, column tile), bumped once when that bucket tile is written
    flags = {}
    tgt_ag_in, tgt_ag_free = 1, ntiles
    tgt_rs = 1

    def f(*key):
        return flags.get(key, 0)

    def bump(*key):
        flags[key] = f(*key) + 1

    slots = {}     # AG: (slot, q, mt) -> shard id
    bufs = {}      # RS: (buf, q, mt, nt) -> (bucket, frozenset(contributors))
    outputs = {}   # AG: (rank, shard, q, mt, nt) -> True ; RS: (bucket, q, mt, nt) -> contributors
    # per CTA: list of tile indices; cursor; phase within a tile
    queues = [[t for t in range(len(tiles)) if t % grid == b] for b in range(grid)]
    cur = [0] * grid
    phase = [0] * grid

    def try_step(b):
        if cur[b] >= len(queues[b]):
            return False
        ti, q, mt, nt = tiles[queues[b][cur[b]]]
        t = tasks[ti]
        if op == AG:
            if phase[b] == 0:       # load A (needs the slot chunk forwarded)
                if t.wait_in[0] >= 0 and f(t.wait_in[0], q, mt) < tgt_ag_in:
                    return False
                shard = t.a_slab if t.a_src == 0 else slots.get((t.a_slab, q, mt))
                if p.direction != "none":
                    assert shard == t.out_idx, f"task {ti} read shard {shard}, wants {t.out_idx}"
                outputs[(t.rank, t.out_idx, q, mt, nt)] = True
                if t.sig_done >= 0:
                    bump(t.sig_done, q, mt)
                phase[b] = 1
                return True
            fwd = nt == 0 and (t.fwd_slot[0] >= 0 or t.fwd_slot[1] >= 0)
            if fwd:
                for j in range(2):
                    if t.fwd_slot[j] >= 0 and t.wait_free[j] >= 0 and f(t.wait_free[j], q, mt) < tgt_ag_free:
                        return False
                for j in range(2):
                    if t.fwd_slot[j] >= 0:
                        slots[(t.fwd_slot[j], q, mt)] = t.out_idx
                        if t.sig_fwd[j] >= 0:
                            bump(t.sig_fwd[j], q, mt)
        else:
            if phase[b] == 0:       # main loop: no cross-CTA dependency
                phase[b] = 1
                return True
            for fl in list(t.wait_in) + [t.wait_free[0]]:
                if fl >= 0 and f(fl, q, mt, nt) < tgt_rs:
                    return False
            if t.a_src == 2:
                contrib = frozenset(range(N))
            else:
                contrib = {t.rank}
                for j in range(2):
                    if t.in_buf[j] >= 0:
                        key = (t.in_buf[j], q, mt, nt)
                        assert key in bufs, f"task {ti} read buffer {key} before any write"
                        bk, cs = bufs[key]
                        assert bk == t.out_idx, f"task {ti} read bucket {bk}, wants {t.out_idx}"
                        assert not (cs & contrib)
                        contrib |= cs
                contrib = frozenset(contrib)
            if t.out_buf >= 0:
                bufs[(t.out_buf, q, mt, nt)] = (t.out_idx, contrib)
            else:
                assert (t.out_idx, q, mt, nt) not in outputs
                outputs[(t.out_idx, q, mt, nt)] = contrib
            if t.sig_done >= 0:
                bump(t.sig_done, q, mt, nt)
        phase[b] = 0
        cur[b] += 1
        return True

    live = list(range(grid))
    while live:
        order = live[:]
        rnd.shuffle(order)
        progressed = False
        for b in order:
            if try_step(b):
                progressed = True
                break
        if not progressed:
            raise AssertionError(f"deadlock: cursors {cur}")
        live = [b for b in range(grid) if cur[b] < len(queues[b])]
    return outputs


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("direction", ["uni", "bidi", "none"])
@pytest.mark.parametrize("chunks", [1, 2, 4])
@pytest.mark.parametrize("grid", [1, 3, 16])
@pytest.mark.parametrize("group", [1, 4])
@pytest.mark.parametrize("in_place", [1, 0])
@pytest.mark.parametrize("order", [0, 2])
def test_protocol_simulation(N, direction, chunks, grid, group, in_place, order):
    if (not in_place or order == 2) and (grid == 3 or group == 1):
        pytest.skip("per-step RS buffers and step-major order: a subset of the grid")
    p = cm.Plan(N, chunks, direction)
    p.set_option(cm.CM_OPT_TILE_GROUP, group)
    p.set_option(cm.CM_OPT_RS_IN_PLACE, in_place)
    p.set_option(cm.CM_OPT_TASK_ORDER, order)
    c = p.chunks
    mtiles, ntiles = 2, 2
    for seed in range(3):
        out = _simulate(p, AG, mtiles, ntiles, grid, seed)
        if direction != "none":
            assert len(out) == N * N * c * mtiles * ntiles
        out = _simulate(p, RS, mtiles, ntiles, grid, seed)
        assert len(out) == N * c * mtiles * ntiles
        assert all(v == frozenset(range(N)) for v in out.values())


@pytest.mark.parametrize("N", [3, 4, 8])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
@pytest.mark.parametrize("chunks", [1, 2])
@pytest.mark.parametrize("grid", [3, 16])
@pytest.mark.parametrize("band", [1, 3])
def test_protocol_simulation_row_bands(N, direction, chunks, grid, band):
    """Row bands reorder tiles inside a task group only: no new wait cycles."""
    p = cm.Plan(N, chunks, direction)
    c = p.chunks
    mtiles, ntiles = 2, 3
    for seed in range(2):
        out = _simulate(p, AG, mtiles, ntiles, grid, seed, band)
        assert len(out) == N * N * c * mtiles * ntiles
        out = _simulate(p, RS, mtiles, ntiles, grid, seed, band)
        assert all(v == frozenset(range(N)) for v in out.values())


@pytest.mark.parametrize("N", [3, 4, 8])
@pytest.mark.parametrize("direction", ["uni", "bidi"])
@pytest.mark.parametrize("grid", [3, 16])
@pytest.mark.parametrize("slabs", [2, 3])
@pytest.mark.parametrize("in_place", [1, 0])
def test_protocol_simulation_column_slabs(N, direction, grid, slabs, in_place):
    """Column slabs (GEMM-RS) run the tile order once per slab of column
    tiles: a bucket tile's predecessor is in the same slab and earlier, so no
    wait cycle, and every bucket still collects every rank once."""
    p = cm.Plan(N, 1, direction)
    p.set_option(cm.CM_OPT_RS_IN_PLACE, in_place)
    mtiles, ntiles = 2, 6
    for seed in range(2):
        out = _simulate(p, RS, mtiles, ntiles, grid, seed, 0, slabs)
        assert len(out) == N * mtiles * ntiles
        assert all(v == frozenset(range(N)) for v in out.values())


@pytest.mark.parametrize("slabs", [1, 2, 3, 6])
def test_column_slab_order_is_a_permutation(slabs):
    p = cm.Plan(8, 2, "uni")
    tasks = p.tasks(RS)
    base = kernel_tile_order(tasks, 2, 3, 6)
    order = kernel_tile_order(tasks, 2, 3, 6, 0, slabs)
    assert sorted(order) == sorted(base)
    # every pass covers only its own slab's columns
    per = len(order) // slabs
    for s_ in range(slabs):
        assert {nt for (_, _, _, nt) in order[s_ * per:(s_ + 1) * per]} == set(range(s_ * 6 // slabs, (s_ + 1) * 6 // slabs))


@pytest.mark.parametrize("band", [0, 1, 2, 3, 5, 100])
def test_row_band_order_is_a_permutation(band):
    p = cm.Plan(8, 2, "uni")
    for op in (AG, RS):
        tasks = p.tasks(op)
        base = kernel_tile_order(tasks, 2, 3, 4)
        order = kernel_tile_order(tasks, 2, 3, 4, band)
        assert sorted(order) == sorted(base)
        if band in (0, 100):
            assert order == base


def test_skip_signal_starves_consumer():
    """Fault injection drops a task's signals: its consumer can never run."""
    p = cm.Plan(4, 1, "uni")
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, (AG << 16) | (1 << 8) | 0)
    with pytest.raises(AssertionError, match="deadlock"):
        _simulate(p, AG, 1, 1, 4, 0)
    p.set_option(cm.CM_OPT_SKIP_SIGNAL, -1)
    _simulate(p, AG, 1, 1, 4, 0)


@pytest.mark.parametrize("op", [AG, RS])
@pytest.mark.parametrize("which", ["wait_in"])
def test_simulation_catches_a_missing_wait(op, which):
    """Planted mistake: a task table without its readiness waits must fail
    the simulation for some interleaving (readiness is the only dependency:
    AG slots are written once, and an in-place bucket's predecessor is its
    only other user)."""
    p = cm.Plan(5, 1, "uni")
    real = p.tasks

    def broken(o):
        ts = real(o)
        for t in ts:
            getattr(t, which)[0] = -1
        return ts

    p.tasks = broken
    caught = 0
    for seed in range(12):
        try:
            _simulate(p, op, 2, 2, 7, seed)
        except AssertionError:
            caught += 1
    assert caught > 0
