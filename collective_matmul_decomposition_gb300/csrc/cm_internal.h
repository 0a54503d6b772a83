// cm_internal.h -- types shared by the planner, the C ABI and the kernel.
#pragma once

#include <cstdint>
#include <vector>

#include "cm.h"

namespace cm {

constexpr int kMaxTasks = CM_MAX_RANKS * CM_MAX_RANKS;   // N tasks per rank at most

// Ring schedule entry of one (rank, step, stream); see cm_plan_step.
struct StepEntry {
    int obj = -1, src = -1, dst = -1;
};

struct Schedule {
    int steps = 0;
    int streams = 1;
    std::vector<StepEntry> e;   // [rank][step][stream]
    StepEntry &at(int N, int r, int i, int s) { return e[(size_t(r) * steps + i) * streams + s]; }
    const StepEntry &at(int N, int r, int i, int s) const {
        return e[(size_t(r) * steps + i) * streams + s];
    }
};

// Flag ids (word = id * chunks + chunk): AG "chunk forwarded into this
// slot" or RS "partial bucket chunk written", one per (rank, step, stream).
enum FlagKind { kFlagReady = 0, kFlagDone = 0 };

struct PlanImpl {
    int N = 1;
    int chunks = 1;
    cm_direction dir = CM_RING_UNI;
    int64_t timeout_ns = 1000000000LL;
    int serial_steps = 0;
    int grid = 0;
    int kernel = 0;         // see CM_OPT_KERNEL
    int static_tiles = 0;   // see CM_OPT_STATIC_TILES
    int tile_group = 4;     // see CM_OPT_TILE_GROUP
    int l2_hints = 0;       // see CM_OPT_L2_HINTS
    int l2_promotion = 3;   // see CM_OPT_L2_PROMOTION
    int row_band = 0;       // see CM_OPT_ROW_BAND
    int bulk_overlap = 1;   // see CM_OPT_BULK_OVERLAP
    int rs_preload = 2;     // see CM_OPT_RS_PRELOAD
    int rs_in_place = 2;    // see CM_OPT_RS_IN_PLACE (2: chosen per call)
    int task_order = 0;     // see CM_OPT_TASK_ORDER
    int rs_epilogue = 0;    // see CM_OPT_RS_EPILOGUE
    int rs_col_slabs = 0;   // see CM_OPT_RS_COL_SLABS
    int rs_bucket_hint = 0; // see CM_OPT_RS_BUCKET_HINT
    int debug_flag_offset = 0;   // see CM_OPT_DEBUG_FLAG_OFFSET (bounds-checked builds)
    int64_t skip_signal = -1;
    Schedule sched[2];                    // per cm_op
    std::vector<cm_task> tasks[2];        // per cm_op, the ring's own execution order
    std::vector<cm_task> tasks_sm[2];     // per cm_op, step-major execution order
    int flag_ids[2] = {0, 0};             // ids used per op (before * chunks)
    std::vector<int> step_begin[2];       // first task index of each step (+ end sentinel)
    std::vector<int> step_begin_sm[2];    // the same for tasks_sm
    // GEMM -> ReduceScatter with one buffer per (rank, stream, step): the same
    // tasks as tasks[CM_OP_GEMM_RS] / tasks_sm[...] (buckets in place) with
    // other buffer indices, in both orders
    std::vector<cm_task> rs_ps, rs_ps_sm;
    std::vector<int> rs_ps_step_begin, rs_ps_step_begin_sm;
};

}  // namespace cm

struct cm_plan_s {
    cm::PlanImpl impl;
};
