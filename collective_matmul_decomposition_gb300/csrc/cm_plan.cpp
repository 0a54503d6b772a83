// cm_plan.cpp -- ring schedules and the task table the persistent kernel runs.
//
// Schedules ("Overlap Communication with Dependent Computation via
// Decomposition in Large Deep Learning Models", section "The idea";
// "Hiding Tensor-Parallel Collectives: AG/RS Overlap in Megatron", sections
// 3 and 5):
//   AG, one ring: rank r multiplies shard (r - i) mod N at step i; it received
//     it from r-1 and forwards it to r+1 until every rank has used it.
//   RS, one ring: rank r adds its product for bucket (r - i - 1) mod N at step
//     i to the partial bucket received from r-1 and forwards it to r+1; at
//     step N-1 that bucket is r's own and is written out.
//   Bidirectional: a = ceil((N-1)/2) clockwise hops, b = floor((N-1)/2)
//     counter-clockwise hops.  AG: the own shard leaves both ways at step 0;
//     rank r uses (r - i) and (r + i) at step i.  RS: the bucket of owner o
//     collects ranks o-a .. o-1 clockwise and o+b .. o+1 counter-clockwise;
//     the owner adds both partials and its own product (the realigning add).
//
// Task table: one task per (rank, step, stream) that multiplies.  Every
// (rank, stream, step) has its own receive slot (AG), written once.  RS
// buckets live either in one fp32 buffer per (bucket, stream) that every
// contributor after the first accumulates into in place (in_buf[0] ==
// out_buf: the kernels add their partial product to it where it lies), or in
// one buffer per (rank, stream, step), written once and read by the next
// rank.  Both tables are built; each call takes one (CM_OPT_RS_IN_PLACE, by
// default from the size of the buckets).  Either way the only dependency is
// readiness: task (r, i) needs what its ring predecessor produced at step
// i-1, and that predecessor is the buffer's only other user at the time.
// Every flag a task waits on is signalled by a task earlier in the table,
// which makes the in-order tile hand-out of the kernels free of deadlock (the
// earliest unfinished tile never waits).
//
// Order.  One ring (uni): rank-blocked --
//   (0,0) | (1,0..1) | (2,0..2) | ... | (N-1,0..N-1) | (0,1..N-1) | (1,2..N-1) | ...
// -- each rank's steps run in order right after its predecessor's, and a
// rank's weight shard W_r is streamed in two runs instead of once per step.
// Bidirectional rings (two predecessors, one each way): stream-blocked --
// the clockwise stream rank-blocked, then the counter-clockwise stream
// rank-blocked over the mirrored ranks -- so W_r is streamed in about four
// runs.  The undecomposed op and the step-serial mode: step-major, and
// inside a step by rank.  CM_OPT_TASK_ORDER may run any ring step-major.
#include <algorithm>
#include <cstring>
#include <new>

#include "cm_internal.h"

namespace cm {
namespace {

inline int md(int a, int N) { return ((a % N) + N) % N; }

void hop_split(int N, int *a, int *b) {
    *a = N / 2;          // ceil((N-1)/2)
    *b = (N - 1) / 2;    // floor((N-1)/2)
}

void build_ag_schedule(PlanImpl &p) {
    const int N = p.N;
    Schedule &s = p.sched[CM_OP_AG_GEMM];
    if (p.dir == CM_RING_NONE) {
        s.steps = 1; s.streams = 1;
        s.e.assign(size_t(N), StepEntry{});
        return;
    }
    if (p.dir == CM_RING_UNI) {
        s.steps = N; s.streams = 1;
        s.e.assign(size_t(N) * N, StepEntry{});
        for (int r = 0; r < N; ++r)
            for (int i = 0; i < N; ++i) {
                StepEntry &e = s.at(N, r, i, 0);
                e.obj = md(r - i, N);
                e.src = i == 0 ? r : md(r - 1, N);
                e.dst = i < N - 1 ? md(r + 1, N) : -1;
            }
        return;
    }
    int a, b;
    hop_split(N, &a, &b);
    s.steps = a + 1; s.streams = 2;
    s.e.assign(size_t(N) * s.steps * 2, StepEntry{});
    for (int r = 0; r < N; ++r) {
        s.at(N, r, 0, 0) = StepEntry{r, r, a >= 1 ? md(r + 1, N) : -1};
        s.at(N, r, 0, 1) = StepEntry{r, r, b >= 1 ? md(r - 1, N) : -1};
        for (int i = 1; i <= a; ++i)
            s.at(N, r, i, 0) = StepEntry{md(r - i, N), md(r - 1, N), i < a ? md(r + 1, N) : -1};
        for (int i = 1; i <= b; ++i)
            s.at(N, r, i, 1) = StepEntry{md(r + i, N), md(r + 1, N), i < b ? md(r - 1, N) : -1};
    }
}

void build_rs_schedule(PlanImpl &p) {
    const int N = p.N;
    Schedule &s = p.sched[CM_OP_GEMM_RS];
    if (p.dir == CM_RING_NONE) {
        s.steps = 1; s.streams = 1;
        s.e.assign(size_t(N), StepEntry{});
        return;
    }
    if (p.dir == CM_RING_UNI) {
        s.steps = N; s.streams = 1;
        s.e.assign(size_t(N) * N, StepEntry{});
        for (int r = 0; r < N; ++r)
            for (int i = 0; i < N; ++i) {
                StepEntry &e = s.at(N, r, i, 0);
                e.obj = md(r - i - 1, N);
                e.src = i == 0 ? -1 : md(r - 1, N);
                e.dst = i < N - 1 ? md(r + 1, N) : -1;
            }
        return;
    }
    int a, b;
    hop_split(N, &a, &b);
    s.steps = a + 1; s.streams = 2;
    s.e.assign(size_t(N) * s.steps * 2, StepEntry{});
    for (int r = 0; r < N; ++r) {
        for (int i = 0; i < a; ++i)
            s.at(N, r, i, 0) = StepEntry{md(r + a - i, N), i == 0 ? -1 : md(r - 1, N), md(r + 1, N)};
        s.at(N, r, a, 0) = StepEntry{r, a >= 1 ? md(r - 1, N) : -1, -1};   // owner
        for (int i = 0; i < b; ++i)
            s.at(N, r, i, 1) = StepEntry{md(r - b + i, N), i == 0 ? -1 : md(r + 1, N), md(r - 1, N)};
    }
}

cm_task blank_task(int rank, int step, int stream) {
    cm_task t;
    std::memset(&t, 0, sizeof t);
    t.rank = int16_t(rank);
    t.out_buf = -1;
    t.in_buf[0] = t.in_buf[1] = -1;
    t.fwd_slot[0] = t.fwd_slot[1] = -1;
    t.wait_in[0] = t.wait_in[1] = -1;
    t.wait_free[0] = t.wait_free[1] = -1;
    t.sig_fwd[0] = t.sig_fwd[1] = -1;
    t.sig_done = -1;
    t.step = int16_t(step);
    t.stream = int16_t(stream);
    return t;
}

struct Ids {
    int N, S;
    // flag id of family `kind` for (rank, step, stream)
    int fid(int kind, int r, int i, int d) const { return ((kind * N + r) * S + i) * 2 + d; }
};

// Position of task (r, i), 0 <= i < S, in the rank-blocked order of a chain
// of S steps over N ranks in which (r, i) waits for (r - 1, i - 1): the
// blocks (r, 0..min(r, S-1)) for r = 0..N-1, then the tails (r, r+1..S-1).
// Whatever a task waits for comes earlier -- in the block before its own, or
// (for a tail, and for rank 0's wrap to rank N-1) in an earlier tail or
// block -- and each rank's tasks form at most two runs.
long rank_blocked_key(int N, int S, int r, int i) {
    long before = 0, first = 0, tails = 0;
    for (int q = 0; q < N; ++q) {
        const int blk = std::min(q, S - 1) + 1;   // tasks of block q
        if (q < r) before += blk;
        first += blk;
        if (q < r) tails += std::max(0, S - 1 - q);
    }
    if (i <= r) return before + i;
    return first + tails + (i - r - 1);
}

// Keys of the stream-blocked order of a bidirectional ring: the clockwise
// stream's tasks in rank-blocked order (their chain runs r-1 -> r), then the
// counter-clockwise stream's in rank-blocked order of the mirrored ranks
// N-1-r (their chain runs r+1 -> r).  Each rank's weight shard is then read
// in at most four runs instead of once per step.  GEMM -> ReduceScatter
// owners (which add both partial buckets) follow the later of their own last
// counter-clockwise task and the counter-clockwise task they wait for, so
// that they usually join their rank's last run.
std::vector<double> stream_blocked_keys(const PlanImpl &p, int op, const std::vector<cm_task> &tasks) {
    const int N = p.N;
    int S[2] = {0, 0};   // steps of each stream's chain (one past the largest step)
    for (const cm_task &t : tasks)
        if (!(op == CM_OP_GEMM_RS && t.out_buf < 0)) S[t.stream] = std::max(S[t.stream], t.step + 1);
    const double off = 1e7;   // the counter-clockwise pass after every clockwise task
    auto key_of = [&](int stream, int r, int i) {
        return stream == 0 ? double(rank_blocked_key(N, S[0], r, i))
                           : off + double(rank_blocked_key(N, S[1], N - 1 - r, i));
    };
    std::vector<double> keys(tasks.size());
    for (size_t j = 0; j < tasks.size(); ++j) {
        const cm_task &t = tasks[j];
        if (op == CM_OP_GEMM_RS && t.out_buf < 0) {   // owner
            if (S[1] == 0) {
                keys[j] = off + t.rank;   // no counter-clockwise stream: after the clockwise pass
            } else {
                const int last = S[1] - 1;
                keys[j] = std::max(key_of(1, t.rank, last), key_of(1, (t.rank + 1) % N, last)) + 0.5;
            }
        } else {
            keys[j] = key_of(t.stream, t.rank, t.step);
        }
    }
    return keys;
}

// Sort `tasks` into execution order -- kind 1: the ring's blocked order
// (rank-blocked for a one-way ring, stream-blocked for a bidirectional one);
// kind 0: step-major -- and fill in the tile groups and the step index `sb`.
void order_and_index(PlanImpl &p, int op, std::vector<cm_task> &tasks, bool blocked, std::vector<int> &sb) {
    if (blocked && p.dir == CM_RING_UNI) {
        const int N = p.N;
        std::stable_sort(tasks.begin(), tasks.end(), [N](const cm_task &x, const cm_task &y) {
            return rank_blocked_key(N, N, x.rank, x.step) < rank_blocked_key(N, N, y.rank, y.step);
        });
    } else if (blocked && p.dir == CM_RING_BIDI) {
        const std::vector<double> keys = stream_blocked_keys(p, op, tasks);
        std::vector<size_t> idx(tasks.size());
        for (size_t j = 0; j < idx.size(); ++j) idx[j] = j;
        std::stable_sort(idx.begin(), idx.end(), [&keys](size_t a, size_t b) { return keys[a] < keys[b]; });
        std::vector<cm_task> sorted;
        sorted.reserve(tasks.size());
        for (size_t j : idx) sorted.push_back(tasks[j]);
        tasks.swap(sorted);
    } else {
        // inside a step, a rank's tasks (its clockwise and counter-clockwise
        // shard or bucket) sit together: they share W_r and form one tile
        // group; tasks of one step never depend on each other
        std::stable_sort(tasks.begin(), tasks.end(), [](const cm_task &x, const cm_task &y) {
            if (x.step != y.step) return x.step < y.step;
            if (x.rank != y.rank) return x.rank < y.rank;
            if (x.stream != y.stream) return x.stream < y.stream;
            return x.out_idx < y.out_idx;
        });
    }
    // tile groups: runs of consecutive same-rank tasks, at most tile_group long
    // (same-rank tasks never depend on each other, so their tiles may interleave)
    // (the step-serial mode launches step by step, so there every task is its own group)
    const int gmax = p.serial_steps ? 1 : p.tile_group;
    for (size_t t = 0; t < tasks.size();) {
        size_t e = t + 1;
        while (e < tasks.size() && int(e - t) < gmax && tasks[e].rank == tasks[t].rank) ++e;
        for (size_t j = t; j < e; ++j) tasks[j].tile_group = int16_t(((e - t) << 8) | (j - t));
        t = e;
    }
    sb.assign(size_t(p.sched[op].steps) + 1, int(tasks.size()));
    for (int t = int(tasks.size()) - 1; t >= 0; --t) sb[tasks[size_t(t)].step] = t;
    for (int i = int(sb.size()) - 2; i >= 0; --i) sb[size_t(i)] = std::min(sb[size_t(i)], sb[size_t(i) + 1]);
}

// Both execution orders of one op's tasks: the ring's own (rank-blocked for a
// one-way ring, stream-blocked for a bidirectional one, step-major for the
// undecomposed op and in the step-serial mode) and the step-major one.
void set_orders(PlanImpl &p, int op, const std::vector<cm_task> &tasks) {
    p.tasks[op] = tasks;
    order_and_index(p, op, p.tasks[op], p.dir != CM_RING_NONE && !p.serial_steps, p.step_begin[op]);
    p.tasks_sm[op] = tasks;
    order_and_index(p, op, p.tasks_sm[op], false, p.step_begin_sm[op]);
}

void build_ag_tasks(PlanImpl &p) {
    const int N = p.N;
    const Schedule &s = p.sched[CM_OP_AG_GEMM];
    const int S = s.steps, D = s.streams;
    Ids ids{N, S};
    p.flag_ids[CM_OP_AG_GEMM] = N * S * 2;
    std::vector<cm_task> tasks;
    auto slot = [&](int r, int d, int step) { return (r * D + d) * S + step; };   // written once
    if (p.dir == CM_RING_NONE) {
        for (int r = 0; r < N; ++r) {
            cm_task t = blank_task(r, 0, 0);
            t.a_src = 0; t.a_slab = 0; t.out_idx = 0;   // all N shards as one row block
            tasks.push_back(t);
        }
    } else {
        for (int r = 0; r < N; ++r) {
            // step 0: the own shard, read in place, forwarded on every stream that has hops
            cm_task t = blank_task(r, 0, 0);
            t.a_src = 0; t.a_slab = int16_t(r); t.out_idx = int16_t(r);
            for (int d = 0; d < D; ++d) {
                const StepEntry &e = s.at(N, r, 0, d);
                if (e.dst < 0) continue;
                t.fwd_slot[d] = int16_t(slot(e.dst, d, 1));
                t.sig_fwd[d] = int16_t(ids.fid(kFlagReady, e.dst, 1, d));
            }
            tasks.push_back(t);
            for (int i = 1; i < S; ++i)
                for (int d = 0; d < D; ++d) {
                    const StepEntry &e = s.at(N, r, i, d);
                    if (e.obj < 0) continue;
                    cm_task u = blank_task(r, i, d);
                    u.a_src = 1; u.a_slab = int16_t(slot(r, d, i)); u.out_idx = int16_t(e.obj);
                    u.wait_in[0] = int16_t(ids.fid(kFlagReady, r, i, d));
                    if (e.dst >= 0) {
                        u.fwd_slot[0] = int16_t(slot(e.dst, d, i + 1));
                        u.sig_fwd[0] = int16_t(ids.fid(kFlagReady, e.dst, i + 1, d));
                    }
                    tasks.push_back(u);
                }
        }
    }
    set_orders(p, CM_OP_AG_GEMM, tasks);
}

void build_rs_tasks(PlanImpl &p, bool in_place) {
    const int N = p.N;
    const Schedule &s = p.sched[CM_OP_GEMM_RS];
    const int S = s.steps, D = s.streams;
    Ids ids{N, S};
    p.flag_ids[CM_OP_GEMM_RS] = N * S * 2;
    std::vector<cm_task> tasks;
    // accumulator buffer that (rank r, stream d, step) reads and a step-i
    // contributor to bucket o writes: one per bucket and stream (in place),
    // or one per (rank, stream, step) (written once)
    auto acc = [&](int r, int d, int step, int bucket) {
        return in_place ? bucket * D + d : (r * D + d) * S + step;
    };
    if (p.dir == CM_RING_NONE) {
        for (int o = 0; o < N; ++o) {
            cm_task t = blank_task(o, 0, 0);
            t.a_src = 2; t.a_slab = 0; t.out_idx = int16_t(o);   // sum over every rank in TMEM
            tasks.push_back(t);
        }
    } else {
        int a = N - 1, b = 0;
        if (p.dir == CM_RING_BIDI) hop_split(N, &a, &b);
        for (int r = 0; r < N; ++r)
            for (int i = 0; i < S; ++i)
                for (int d = 0; d < D; ++d) {
                    const StepEntry &e = s.at(N, r, i, d);
                    if (e.obj < 0) continue;
                    cm_task t = blank_task(r, i, d);
                    t.a_src = 0; t.a_slab = int16_t(r * N + e.obj); t.out_idx = int16_t(e.obj);
                    t.sig_done = int16_t(ids.fid(kFlagDone, r, i, d));
                    const bool owner = e.dst < 0;
                    const int o = e.obj;
                    if (!owner) {
                        // partial bucket goes to the next rank of this stream
                        // (in place: the bucket's one buffer, which this
                        // task starts at step 0 and adds to after that)
                        t.out_buf = int16_t(acc(e.dst, d, i + 1, o));
                        if (i > 0) {
                            t.in_buf[0] = int16_t(acc(r, d, i, o));
                            t.wait_in[0] = int16_t(ids.fid(kFlagDone, e.src, i - 1, d));
                        }
                    } else if (p.dir == CM_RING_UNI) {
                        if (i > 0) {
                            t.in_buf[0] = int16_t(acc(r, 0, i, o));
                            t.wait_in[0] = int16_t(ids.fid(kFlagDone, e.src, i - 1, 0));
                        }
                    } else {
                        // realigning addition: clockwise partial arrived at step a,
                        // counter-clockwise partial at step b
                        if (a >= 1) {
                            t.in_buf[0] = int16_t(acc(r, 0, a, o));
                            t.wait_in[0] = int16_t(ids.fid(kFlagDone, md(r - 1, N), a - 1, 0));
                        }
                        if (b >= 1) {
                            t.in_buf[1] = int16_t(acc(r, 1, b, o));
                            t.wait_in[1] = int16_t(ids.fid(kFlagDone, md(r + 1, N), b - 1, 1));
                        }
                    }
                    tasks.push_back(t);
                }
    }
    if (in_place) {
        set_orders(p, CM_OP_GEMM_RS, tasks);
    } else {
        p.rs_ps = tasks;
        order_and_index(p, CM_OP_GEMM_RS, p.rs_ps, p.dir != CM_RING_NONE && !p.serial_steps, p.rs_ps_step_begin);
        p.rs_ps_sm = tasks;
        order_and_index(p, CM_OP_GEMM_RS, p.rs_ps_sm, false, p.rs_ps_step_begin_sm);
    }
}

// Bounds-checked builds: the planted out-of-range done-signal ids of
// CM_OPT_DEBUG_FLAG_OFFSET.
void apply_debug_offset(PlanImpl &p) {
    if (p.debug_flag_offset <= 0) return;
    for (auto *v : {&p.tasks[CM_OP_GEMM_RS], &p.tasks_sm[CM_OP_GEMM_RS], &p.rs_ps, &p.rs_ps_sm})
        for (cm_task &t : *v)
            if (t.sig_done >= 0) t.sig_done = int16_t(t.sig_done + p.debug_flag_offset);
}

void apply_skip(PlanImpl &p) {
    if (p.skip_signal < 0) return;
    const int op = int((p.skip_signal >> 16) & 0xff);
    const int rank = int((p.skip_signal >> 8) & 0xff);
    const int step = int(p.skip_signal & 0xff);
    if (op > 1) return;
    std::vector<std::vector<cm_task> *> tables = {&p.tasks[op], &p.tasks_sm[op]};
    if (op == CM_OP_GEMM_RS) {
        tables.push_back(&p.rs_ps);
        tables.push_back(&p.rs_ps_sm);
    }
    for (auto *v : tables)
        for (cm_task &t : *v)
            if (t.rank == rank && t.step == step) {
                t.sig_fwd[0] = t.sig_fwd[1] = -1;
                t.sig_done = -1;
            }
}

}  // namespace

void rebuild(PlanImpl &p) {
    build_ag_schedule(p);
    build_rs_schedule(p);
    build_ag_tasks(p);
    build_rs_tasks(p, true);
    build_rs_tasks(p, false);
    apply_skip(p);
    apply_debug_offset(p);
}

}  // namespace cm

extern "C" {

cm_status cm_plan(int n_ranks, int chunks, cm_direction dir, cm_plan_t *out) {
    if (!out) return CM_ERR_INVALID_ARG;
    *out = nullptr;
    if (n_ranks < 1 || n_ranks > CM_MAX_RANKS || chunks < 1 || chunks > CM_MAX_CHUNKS)
        return CM_ERR_INVALID_ARG;
    if (dir != CM_RING_UNI && dir != CM_RING_BIDI && dir != CM_RING_NONE) return CM_ERR_INVALID_ARG;
    cm_plan_s *p = new (std::nothrow) cm_plan_s();
    if (!p) return CM_ERR_INVALID_ARG;
    p->impl.N = n_ranks;
    p->impl.chunks = dir == CM_RING_NONE ? 1 : chunks;
    p->impl.dir = dir;
    try {
        cm::rebuild(p->impl);
    } catch (...) {
        delete p;
        return CM_ERR_INVALID_ARG;
    }
    *out = p;
    return CM_OK;
}

cm_status cm_plan_destroy(cm_plan_t plan) {
    delete plan;
    return CM_OK;
}

int cm_plan_steps(cm_plan_t plan, cm_op op) {
    if (!plan || (op != CM_OP_AG_GEMM && op != CM_OP_GEMM_RS)) return -1;
    return plan->impl.sched[op].steps;
}

cm_status cm_plan_step(cm_plan_t plan, cm_op op, int rank, int step, int stream,
                       int *obj, int *src, int *dst) {
    if (!plan || (op != CM_OP_AG_GEMM && op != CM_OP_GEMM_RS)) return CM_ERR_INVALID_ARG;
    const cm::PlanImpl &p = plan->impl;
    const cm::Schedule &s = p.sched[op];
    if (rank < 0 || rank >= p.N || step < 0 || step >= s.steps || stream < 0 || stream > 1)
        return CM_ERR_INVALID_ARG;
    cm::StepEntry e;
    if (stream < s.streams) e = s.at(p.N, rank, step, stream);
    if (obj) *obj = e.obj;
    if (src) *src = e.src;
    if (dst) *dst = e.dst;
    return CM_OK;
}

int cm_plan_tasks(cm_plan_t plan, cm_op op, cm_task *out, int capacity) {
    if (!plan || (op != CM_OP_AG_GEMM && op != CM_OP_GEMM_RS)) return -1;
    const cm::PlanImpl &pl = plan->impl;
    const bool ps = op == CM_OP_GEMM_RS && pl.rs_in_place == 0;   // per-step table; 1 and 2 list the in-place one
    const auto &t = pl.task_order == 2 ? (ps ? pl.rs_ps_sm : pl.tasks_sm[op]) : (ps ? pl.rs_ps : pl.tasks[op]);
    for (int i = 0; i < capacity && i < int(t.size()); ++i) out[i] = t[size_t(i)];
    return int(t.size());
}

cm_status cm_plan_set_option(cm_plan_t plan, cm_option option, int64_t value) {
    if (!plan) return CM_ERR_INVALID_ARG;
    cm::PlanImpl &p = plan->impl;
    switch (option) {
        case CM_OPT_TIMEOUT_NS:
            if (value <= 0) return CM_ERR_INVALID_ARG;
            p.timeout_ns = value;
            return CM_OK;
        case CM_OPT_SERIAL_STEPS:
            p.serial_steps = value != 0;
            try {
                cm::rebuild(p);   // the step-serial mode runs the table in step-major order
            } catch (...) {
                return CM_ERR_INVALID_ARG;
            }
            return CM_OK;
        case CM_OPT_GRID:
            if (value < 0) return CM_ERR_INVALID_ARG;
            p.grid = int(value);
            return CM_OK;
        case CM_OPT_KERNEL:
            if (value < 0 || value > 2) return CM_ERR_INVALID_ARG;
            p.kernel = int(value);
            return CM_OK;
        case CM_OPT_TILE_GROUP:
            if (value < 1 || value > 8) return CM_ERR_INVALID_ARG;
            p.tile_group = int(value);
            try {
                cm::rebuild(p);
            } catch (...) {
                return CM_ERR_INVALID_ARG;
            }
            return CM_OK;
        case CM_OPT_L2_HINTS:
            if (value < 0 || value > 0xff) return CM_ERR_INVALID_ARG;
            p.l2_hints = int(value);
            return CM_OK;
        case CM_OPT_BULK_OVERLAP:
            if (value != 0 && value != 1) return CM_ERR_INVALID_ARG;
            p.bulk_overlap = int(value);
            return CM_OK;
        case CM_OPT_RS_PRELOAD:
            if (value < 0 || value > 3) return CM_ERR_INVALID_ARG;
            p.rs_preload = int(value);
            return CM_OK;
        case CM_OPT_ROW_BAND:
            if (value < 0 || value > 4096) return CM_ERR_INVALID_ARG;
            p.row_band = int(value);
            return CM_OK;
        case CM_OPT_L2_PROMOTION:
            if (value < 0 || value > 3) return CM_ERR_INVALID_ARG;
            p.l2_promotion = int(value);
            return CM_OK;
        case CM_OPT_STATIC_TILES:
            p.static_tiles = value != 0;
            return CM_OK;
        case CM_OPT_DEBUG_FLAG_OFFSET:
#ifdef CM_DEBUG_BOUNDS
            if (value < 0 || value > 4096) return CM_ERR_INVALID_ARG;
            p.debug_flag_offset = int(value);
            try {
                cm::rebuild(p);
            } catch (...) {
                return CM_ERR_INVALID_ARG;
            }
            return CM_OK;
#else
            return CM_ERR_INVALID_ARG;   // a testing aid of the bounds-checked build only
#endif
        case CM_OPT_RS_BUCKET_HINT:
            if (value < 0 || value > 3) return CM_ERR_INVALID_ARG;
            p.rs_bucket_hint = int(value);
            return CM_OK;
        case CM_OPT_RS_COL_SLABS:
            if (value < 0 || value > 64) return CM_ERR_INVALID_ARG;
            p.rs_col_slabs = int(value);
            return CM_OK;
        case CM_OPT_RS_EPILOGUE:
            if (value < 0 || value > 3) return CM_ERR_INVALID_ARG;
            p.rs_epilogue = int(value);
            return CM_OK;
        case CM_OPT_TASK_ORDER:
            if (value < 0 || value > 2) return CM_ERR_INVALID_ARG;
            p.task_order = int(value);
            return CM_OK;
        case CM_OPT_RS_IN_PLACE:   // both task tables are built; each call picks one
            if (value < 0 || value > 2) return CM_ERR_INVALID_ARG;
            p.rs_in_place = int(value);
            return CM_OK;
        case CM_OPT_SKIP_SIGNAL:
            p.skip_signal = value < 0 ? -1 : value;
            try {
                cm::rebuild(p);
            } catch (...) {
                return CM_ERR_INVALID_ARG;
            }
            return CM_OK;
    }
    return CM_ERR_INVALID_ARG;
}

}  // extern "C"
