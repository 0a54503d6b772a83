// cm_kernel_common.cuh -- tile decoding, flags and bounded waits shared by
// the single-CTA and the CTA-pair persistent kernels.
#pragma once

#include "cm_device.cuh"
#include "cm_kernel.cuh"

namespace cm {
namespace kc {
namespace {   // internal linkage: each kernel translation unit has its own copy

using namespace dev;

struct TileCoord {
    int task, q, mt, nt;
};

// Linear tile index -> (task, chunk, row tile, column tile) of one CTA (or
// one CTA pair).  Tiles run task group by task group (see cm_task.tile_group);
// inside a group the order is chunk, row band, column tile, row tile of the
// band.  The group's row tiles (task by task) are cut into bands of
// `row_band` row tiles (0: one band); each band runs through every column
// tile before the next band starts, so the tiles running together share one
// block of weight columns (W_r of the group's rank) and one band of A rows.
// With column slabs (col_slabs > 1) all of that runs once per slab of
// ntiles / col_slabs column tiles, slab after slab: the tasks' buckets are
// then touched one slab at a time.
__device__ __forceinline__ TileCoord decode(const KParams &p, int t) {
    TileCoord c;
    const int slabs = p.col_slabs > 1 ? p.col_slabs : 1;
    const int nts = p.ntiles / slabs;                  // column tiles of one slab
    const int tpt = p.tiles_per_task / slabs;          // tiles of one task in one slab
    const int slab = t / ((p.task_end - p.task_begin) * tpt);
    t -= slab * (p.task_end - p.task_begin) * tpt;
    const int task = p.task_begin + t / tpt;
    const int16_t grp = p.tasks[task].tile_group;
    const int gsize = grp >> 8, gpos = grp & 0xff;
    const int gfirst = task - gpos;
    int u = t - (gfirst - p.task_begin) * tpt;   // tile index inside the group
    const int rows = gsize * p.mtiles_c;          // row tiles of the group
    const int per_q = rows * nts;
    c.q = u / per_q;
    u -= c.q * per_q;
    if (p.q_only >= 0) c.q = p.q_only;   // one chunk per launch: u never reaches a second one
    const int band = p.row_band > 0 && p.row_band < rows ? p.row_band : rows;
    const int full = rows / band;
    const int in_full = full * band * nts;
    int b0, bs;   // first row tile and row tiles of this tile's band
    if (u < in_full) {
        const int b = u / (band * nts);
        b0 = b * band;
        bs = band;
        u -= b * band * nts;
    } else {
        b0 = full * band;
        bs = rows - b0;
        u -= in_full;
    }
    const int g = u / bs;
    const int rho = b0 + (u - g * bs);
    const int off = rho / p.mtiles_c;
    c.mt = rho - off * p.mtiles_c;
    c.task = gfirst + off;
    c.nt = slab * nts + g;
    return c;
}

// Readiness counter of flag `id` for the tile region a task reads or writes:
// AG, one per (id, chunk, row tile) -- the shard rows of one row tile arrive
// together (every column tile of the forwarding task sends a slice of them);
// RS, one per (id, chunk, row tile, column tile) -- the bucket tile a task
// adds to depends only on its predecessor's same tile.
#ifdef CM_DEBUG_BOUNDS
constexpr bool kCheckBounds = true;
#else
constexpr bool kCheckBounds = false;
#endif
// Word of the status block that a rejected flag access is sent to (debug
// builds); no wait on it ever completes, so its waiters see the failure.
constexpr int kSinkWord = 48;

// Debug builds: record that a computed index fell outside its buffer
// (CM_ERR_BOUNDS, with task, chunk and which index), unless an earlier
// failure was recorded.  The caller then skips the access.
__device__ __noinline__ void report_bounds(const KParams &p, uint32_t site, int task, int q) {
    if (atomicCAS(p.status, 0u, uint32_t(CM_ERR_BOUNDS)) == 0u) {
        p.status[1] = uint32_t(task);
        p.status[2] = uint32_t(q);
        p.status[3] = site;
        __threadfence();
    }
}

// true if `ok`; in debug builds a false `ok` is reported first.  Release
// builds compile the check away (always true).
__device__ __forceinline__ bool in_bounds(const KParams &p, bool ok, uint32_t site, int task, int q) {
    if (!kCheckBounds || ok) return true;
    report_bounds(p, site, task, q);
    return false;
}

__device__ __forceinline__ uint32_t *flag_ptr(const KParams &p, int id, int q, int mt, int nt) {
    size_t w = (size_t(id) * size_t(p.chunks) + size_t(q)) * size_t(p.mtiles_c) + size_t(mt);
    if (p.op == 1) w = w * size_t(p.ntiles) + size_t(nt);
    if (!in_bounds(p, id >= 0 && q >= 0 && q < p.chunks && int64_t(w) < p.flag_words, kSiteBoundsFlag, id, q))
        return p.status + kSinkWord;
    return p.flags + w;
}

__device__ __forceinline__ int kslices(const KParams &p, const cm_task &tk) {
    return tk.a_src == 2 ? p.kblocks * p.N : p.kblocks;
}

__device__ __noinline__ void report(const KParams &p, uint32_t site, int task, int q) {
    if (atomicCAS(p.status, 0u, uint32_t(CM_ERR_TIMEOUT)) == 0u) {
        p.status[1] = uint32_t(task);
        p.status[2] = uint32_t(q);
        p.status[3] = site;
        __threadfence();
    }
}

// Bounded wait on an mbarrier phase (cluster-scope acquire when `cluster`).
// Returns false -- and marks the CTA as aborting -- if the bound expires, the
// CTA is already aborting, or another CTA has reported a failure.
template <bool kCluster>
__device__ bool wait_mbar(const KParams &p, volatile int *abort, uint64_t *bar, uint32_t parity, uint32_t site,
                          int task, int q) {
    auto try_once = [&]() { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (try_once()) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (try_once()) return true;
        if ((it & 63u) == 0u) {
            if (*abort) return false;
            if ((it & 1023u) == 0u && ld_relaxed(p.status) != 0u) {
                *abort = 1;
                return false;
            }
            if (globaltimer() - t0 > p.timeout_ns) {
                report(p, site, task, q);
                *abort = 1;
                return false;
            }
        }
    }
}

// Bounded wait for a cross-CTA counter to reach `target` (gpu-scope acquire).
__device__ bool wait_flag(const KParams &p, volatile int *abort, const uint32_t *f, uint32_t target, uint32_t site,
                          int task, int q) {
    if (ld_acquire(f) >= target) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (ld_acquire(f) >= target) return true;
        if ((it & 15u) == 0u) {
            if (*abort) return false;
            if (ld_relaxed(p.status) != 0u) {
                *abort = 1;
                return false;
            }
            if (globaltimer() - t0 > p.timeout_ns) {
                report(p, site, task, q);
                *abort = 1;
                return false;
            }
        }
        __nanosleep(64);
    }
}

// Wait that ignores the abort flag (only to drain work already issued).
template <bool kCluster>
__device__ void drain_mbar(const KParams &p, uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!(kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)))
        if (globaltimer() - t0 > p.timeout_ns) break;
}

__device__ __forceinline__ void add4(float *v, const float4 &a) {
    v[0] += a.x;
    v[1] += a.y;
    v[2] += a.z;
    v[3] += a.w;
}

}  // namespace
}  // namespace kc
}  // namespace cm
