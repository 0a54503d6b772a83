// cm_cost.cpp -- the peak-rate cost model that decides, per operation,
// whether to decompose and with which ring.
//
// "Overlap Communication with Dependent Computation via Decomposition in
// Large Deep Learning Models", section "The idea" (knowing when to decline)
// and section "What it costs": the decomposed ring drives one link per
// direction instead of the full collective topology, so the rewrite loses
// whenever a step's compute is shorter than its (slower) transfer; a model
// built from peak rates decides per operation whether to rewrite.  A bidirectional ring's pre-shift
// and realigning addition are charged as unoverlappable.  "Hiding
// Tensor-Parallel Collectives: AG/RS Overlap in Megatron", section 6: more
// chunks shorten the exposed first transfer but add a per-chunk cost.
//
// The model follows one rank (all ranks are alike).  Resources: the rank's
// compute (serial), and one outgoing link per ring direction (serial).
// Every chunk of every step is an event:
//   AG  chunk q of the shard used at step i arrives when the neighbour has
//       forwarded it -- the neighbour forwards a chunk as soon as it has it
//       and its link is free -- and is multiplied once it has arrived and
//       the compute is free.
//   RS  the partial products run back to back on the compute (they need
//       nothing received); the sum for chunk q of step i is ready once its
//       product is done and the received partial bucket chunk has arrived,
//       and is forwarded when the link is free.  The last step's sum is the
//       rank's own bucket.
// Every transfer (every chunk on every hop) also pays a fixed cost that holds
// its link (the flag round trip and launch of one message), which is what
// makes more chunks cost something.  The
// native alternative runs the collective at its own bandwidth, then the
// undecomposed GEMM, with no overlap.  All rates are peak rates supplied by
// the caller (measured).
#include <algorithm>
#include <cmath>
#include <vector>

#include "cm.h"

namespace {

struct Rates {
    double flop_per_us;   // rank's GEMM rate
    double ring_b_per_us; // one ring link, one direction
    double coll_b_per_us; // native collective bandwidth
    double hop_us;        // latency of one transfer (flag round trip)
    double mem_b_per_us;  // rank's local memory bandwidth (realigning add)
};

bool rates_ok(const cm_rates *r) {
    return r && std::isfinite(r->gemm_tflops) && r->gemm_tflops > 0 && std::isfinite(r->ring_gbs) &&
           r->ring_gbs > 0 && std::isfinite(r->coll_gbs) && r->coll_gbs > 0 && std::isfinite(r->hop_us) &&
           r->hop_us >= 0 && std::isfinite(r->mem_gbs) && r->mem_gbs > 0;
}

Rates to_rates(const cm_rates *r) {
    return {r->gemm_tflops * 1e6, r->ring_gbs * 1e3, r->coll_gbs * 1e3, r->hop_us, r->mem_gbs * 1e3};
}

// Shards used by one rank, step by step, with the link (0 = clockwise, 1 =
// counter-clockwise) each arrived on.  Step 0 is the own shard (link -1).
std::vector<std::vector<int>> ag_steps(int N, cm_direction dir) {
    std::vector<std::vector<int>> steps;
    steps.push_back({-1});
    if (dir == CM_RING_UNI) {
        for (int i = 1; i < N; ++i) steps.push_back({0});
    } else {
        const int a = N / 2, b = (N - 1) / 2;   // clockwise / counter-clockwise hops
        for (int i = 1; i <= a; ++i) {
            std::vector<int> s{0};
            if (i <= b) s.push_back(1);
            steps.push_back(s);
        }
    }
    return steps;
}

// AG: chunk transfers per link run back to back; a hop-i chunk can leave only
// after its hop-(i-1) copy arrived.  Compute takes the arrivals in step order.
double ag_time(const Rates &R, int N, int c, cm_direction dir, double m, double K, double n) {
    const double t_c = 2.0 * m * K * n / R.flop_per_us / c;   // one chunk's GEMM
    const double t_x = m * K * 2.0 / R.ring_b_per_us / c;     // one chunk over one link
    const auto steps = ag_steps(N, dir);
    double link_free[2] = {0.0, 0.0};
    // arrival of chunk q over link l at hop h (hop 1 = the first arrival)
    std::vector<std::vector<double>> prev(2, std::vector<double>(size_t(c), 0.0));   // own shard: resident
    std::vector<std::vector<double>> arr(2, std::vector<double>(size_t(c), 0.0));
    double comp = 0.0;
    for (size_t i = 0; i < steps.size(); ++i) {
        if (i > 0) {
            for (int l = 0; l < 2; ++l) {
                bool used = false;
                for (int s : steps[i]) used |= s == l;
                if (!used) continue;
                for (int q = 0; q < c; ++q) {
                    const double start = std::max(prev[size_t(l)][size_t(q)], link_free[l]);
                    link_free[l] = start + t_x + R.hop_us;
                    arr[size_t(l)][size_t(q)] = link_free[l];
                }
                prev[size_t(l)] = arr[size_t(l)];
            }
        }
        for (int s : steps[i])
            for (int q = 0; q < c; ++q) {
                const double ready = s < 0 ? 0.0 : arr[size_t(s)][size_t(q)];
                comp = std::max(comp, ready) + t_c;
            }
    }
    return comp;
}

// RS: one ring carries every bucket N-1 hops; a bidirectional ring splits
// each bucket's contributions into a clockwise run of a hops and a
// counter-clockwise run of b hops, and the owner adds both (realigning add).
double rs_time(const Rates &R, int N, int c, cm_direction dir, double M, double k, double n) {
    const double rows = M / N;
    const double t_c = 2.0 * rows * k * n / R.flop_per_us / c;   // one chunk's partial GEMM
    const double t_x = rows * n * 4.0 / R.ring_b_per_us / c;     // one fp32 chunk over one link
    const int a = dir == CM_RING_UNI ? N - 1 : N / 2;            // clockwise hops of a bucket
    const int b = dir == CM_RING_UNI ? 0 : (N - 1) / 2;          // counter-clockwise hops
    // Contributions in compute order: a clockwise run of a steps and a
    // counter-clockwise run of b steps, one of each per step while both last,
    // then the owner's own.  The partial GEMMs run back to back (they need
    // nothing received); a contribution's sum is ready once its GEMM is done
    // and the partial bucket it adds to has arrived, and is then forwarded.
    double gemm = 0.0, done = 0.0, link_free[2] = {0.0, 0.0};
    std::vector<std::vector<double>> arr(2, std::vector<double>(size_t(c), 0.0));   // bucket chunk at this rank
    auto contribute = [&](int l, bool first) {
        for (int q = 0; q < c; ++q) {
            gemm += t_c;
            const double sum = first ? gemm : std::max(gemm, arr[size_t(l)][size_t(q)]);
            const double start = std::max(sum, link_free[l]);
            link_free[l] = start + t_x + R.hop_us;
            arr[size_t(l)][size_t(q)] = link_free[l];
        }
    };
    const int steps = std::max(a, b);
    for (int i = 0; i < steps; ++i) {
        if (i < a) contribute(0, i == 0);
        if (i < b) contribute(1, i == 0);
    }
    // owner: its own product plus the received partial(s)
    for (int q = 0; q < c; ++q) {
        gemm += t_c;
        double ready = gemm;
        if (a > 0) ready = std::max(ready, arr[0][size_t(q)]);
        if (b > 0) ready = std::max(ready, arr[1][size_t(q)]);
        done = std::max(done, ready);
    }
    if (b > 0) done += 3.0 * rows * n * 4.0 / R.mem_b_per_us;   // realigning add: read two partials, write one
    return done;
}

double native_time(const Rates &R, int N, int op, double rows, double K, double n) {
    if (op == CM_OP_AG_GEMM) {   // AllGather, then the gathered GEMM
        return (N - 1) * rows * K * 2.0 / R.coll_b_per_us + 2.0 * N * rows * K * n / R.flop_per_us;
    }
    // full partial product, then ReduceScatter of fp32 partial buckets
    return 2.0 * rows * K * n / R.flop_per_us + (N - 1) * (rows / N) * n * 4.0 / R.coll_b_per_us;
}

}  // namespace

extern "C" cm_status cm_cost_estimate(int n_ranks, int chunks, cm_direction dir, cm_op op, int64_t rows, int64_t K,
                                      int64_t n, const cm_rates *rates, double *us) {
    if (!us || !rates_ok(rates) || n_ranks < 1 || n_ranks > CM_MAX_RANKS || chunks < 1 || chunks > CM_MAX_CHUNKS ||
        rows < 1 || K < 1 || n < 1 || (op != CM_OP_AG_GEMM && op != CM_OP_GEMM_RS) ||
        (dir != CM_RING_UNI && dir != CM_RING_BIDI && dir != CM_RING_NONE))
        return CM_ERR_INVALID_ARG;
    if (op == CM_OP_GEMM_RS && rows % n_ranks != 0) return CM_ERR_SHAPE;
    const Rates R = to_rates(rates);
    const int N = n_ranks;
    if (dir == CM_RING_NONE || N == 1) {
        *us = native_time(R, N, op, double(rows), double(K), double(n));
        return CM_OK;
    }
    *us = op == CM_OP_AG_GEMM ? ag_time(R, N, chunks, dir, double(rows), double(K), double(n))
                              : rs_time(R, N, chunks, dir, double(rows), double(K), double(n));
    return CM_OK;
}

extern "C" cm_status cm_plan_choose(int n_ranks, cm_op op, int64_t rows, int64_t K, int64_t n, const cm_rates *rates,
                                    int max_chunks, int *chunks, cm_direction *dir, double *us) {
    if (!chunks || !dir || max_chunks < 1 || max_chunks > CM_MAX_CHUNKS) return CM_ERR_INVALID_ARG;
    double best = 0.0;
    cm_status st = cm_cost_estimate(n_ranks, 1, CM_RING_NONE, op, rows, K, n, rates, &best);
    if (st != CM_OK) return st;
    int bc = 1;
    cm_direction bd = CM_RING_NONE;
    // chunk rows: the shard (AG) or bucket (RS) must split evenly
    const int64_t unit = op == CM_OP_AG_GEMM ? rows : rows / n_ranks;
    for (int d = 0; d < 2 && n_ranks > 1; ++d) {
        const cm_direction cand = d == 0 ? CM_RING_UNI : CM_RING_BIDI;
        for (int c = 1; c <= max_chunks; c *= 2) {
            if (unit % c != 0) continue;
            double t = 0.0;
            st = cm_cost_estimate(n_ranks, c, cand, op, rows, K, n, rates, &t);
            if (st != CM_OK) return st;
            if (t < best * (1.0 - 1e-9)) {   // ties (up to rounding) keep the simpler choice
                best = t;
                bc = c;
                bd = cand;
            }
        }
    }
    *chunks = bc;
    *dir = bd;
    if (us) *us = best;
    return CM_OK;
}

// One Einsum that offers both collectives ("Overlap Communication with
// Dependent Computation via Decomposition in Large Deep Learning Models",
// section "The idea", knowing when to decline: where one Einsum has both a
// gathered input and a scattered output, the same cost model also decides
// which of the two collectives to turn into the ring).  Per
// rank: its A operand is the AllGather of N row shards [m, K], it multiplies
// that [N*m, K] by its [K, n] weight, and the [N*m, n] result is summed over
// the ranks and scattered, bucket o being rows o*m.. of the sum.  Only one
// collective can become the ring (the loop runs over input shards or over
// output buckets); the other stays native:
//   gather decomposed:  the AG ring, then the native ReduceScatter of the
//                       fp32 result;
//   scatter decomposed: the native AllGather, then the RS ring;
//   neither:            native AllGather, GEMM, native ReduceScatter.
extern "C" cm_status cm_einsum_cost(int n_ranks, int chunks, cm_direction dir, int decompose, int64_t m, int64_t K,
                                    int64_t n, const cm_rates *rates, double *us) {
    if (!us || !rates_ok(rates) || n_ranks < 1 || n_ranks > CM_MAX_RANKS || chunks < 1 || chunks > CM_MAX_CHUNKS ||
        m < 1 || K < 1 || n < 1 || (dir != CM_RING_UNI && dir != CM_RING_BIDI && dir != CM_RING_NONE) ||
        (decompose != -1 && decompose != CM_OP_AG_GEMM && decompose != CM_OP_GEMM_RS))
        return CM_ERR_INVALID_ARG;
    const Rates R = to_rates(rates);
    const int N = n_ranks;
    const double dm = double(m), dK = double(K), dn = double(n);
    const double ag_native = (N - 1) * dm * dK * 2.0 / R.coll_b_per_us;   // gather of N-1 shards
    const double rs_native = (N - 1) * dm * dn * 4.0 / R.coll_b_per_us;   // scatter of N-1 fp32 buckets
    const double gemm = 2.0 * N * dm * dK * dn / R.flop_per_us;
    const bool ring = dir != CM_RING_NONE && N > 1;
    if (decompose == CM_OP_AG_GEMM && ring) {
        *us = ag_time(R, N, chunks, dir, dm, dK, dn) + rs_native;
    } else if (decompose == CM_OP_GEMM_RS && ring) {
        *us = ag_native + rs_time(R, N, chunks, dir, double(N) * dm, dK, dn);
    } else {
        *us = ag_native + gemm + rs_native;
    }
    return CM_OK;
}

extern "C" cm_status cm_plan_choose_einsum(int n_ranks, int64_t m, int64_t K, int64_t n, const cm_rates *rates,
                                           int max_chunks, int *decompose, int *chunks, cm_direction *dir,
                                           double *us) {
    if (!decompose || !chunks || !dir || max_chunks < 1 || max_chunks > CM_MAX_CHUNKS) return CM_ERR_INVALID_ARG;
    double best = 0.0;
    cm_status st = cm_einsum_cost(n_ranks, 1, CM_RING_NONE, -1, m, K, n, rates, &best);
    if (st != CM_OK) return st;
    int bw = -1, bc = 1;
    cm_direction bd = CM_RING_NONE;
    // candidates in order of simplicity: the gather, then the scatter; one-way
    // before two-way rings; fewer chunks first (a chunk must split the shard,
    // or the bucket -- also m rows -- evenly).  Ties keep the simpler choice.
    for (int which : {int(CM_OP_AG_GEMM), int(CM_OP_GEMM_RS)})
        for (int d = 0; d < 2 && n_ranks > 1; ++d) {
            const cm_direction cand = d == 0 ? CM_RING_UNI : CM_RING_BIDI;
            for (int c = 1; c <= max_chunks; c *= 2) {
                if (m % c != 0) continue;
                double t = 0.0;
                st = cm_einsum_cost(n_ranks, c, cand, which, m, K, n, rates, &t);
                if (st != CM_OK) return st;
                if (t < best * (1.0 - 1e-9)) {
                    best = t;
                    bw = which;
                    bc = c;
                    bd = cand;
                }
            }
        }
    *decompose = bw;
    *chunks = bc;
    *dir = bd;
    if (us) *us = best;
    return CM_OK;
}
