// cm_api.cu -- the C ABI: argument checks, workspace layout, TMA tensor maps
// and the launch of the persistent kernel.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "cm_internal.h"
#include "cm_kernel.cuh"

namespace cm {
namespace {

constexpr size_t kStatusBytes = 256;   // status word at 0, tile counters at kCounterOff
constexpr size_t kCounterOff = 64;
// CM_OPT_RS_PRELOAD automatic choice, by the K slices of a tile: up to
// kPreloadAllKSlices the whole received bucket is preloaded (the epilogue
// sets the pace there: 4 slices measured 13 % faster); beyond that none
// (24 to 112 slices measured 2-7 % slower with all or half preloaded: a
// preloaded tile cannot start its MMAs before the bucket is complete).
constexpr int64_t kPreloadAllKSlices = 8;

// CM_OPT_RS_EPILOGUE: 1 = every epilogue warp on every tile, TMA copies
// through shared memory; 2 = two warp groups, one per accumulator, with
// vector reductions; 3 = every epilogue warp on every tile, vector
// reductions; 0 = automatic.  Returns the kernel's mode (KParams::rs_epi):
// the option value less one.
// The automatic choice, measured over the MLP sweep (h=8192, ffn=28672,
// s=8192) and the GPT-3 attention-out GEMM-RS with both interleaved: two
// groups were 2-6 % faster on one-way rings of 8 and 16 ranks with at least
// 28 K slices per tile and on two-way rings of 16 ranks; the TMA epilogue
// was as fast or faster everywhere else (6-11 % on the GPT-3 layer, 24 K
// slices; 1-3 % at 4 ranks and on two-way rings of 8).  Those tiles read
// nothing back (buckets in place, pipelined partials); where every tile
// loads its input -- buckets in per-step buffers, Cannon's chained
// accumulator (q = 4: 1.17 against 1.37 ms) -- the TMA epilogue is used.
// Every warp with vector reductions (3) measured in between: GPT-3
// attention-out 0.462 ms against 0.440 (TMA) and 0.475 (groups), within
// 1.5 % of the better of the other two on the MLP sweep; it is never chosen
// automatically.
// reads_inputs: the tiles of the call load a received bucket in the epilogue.
int rs_epi_mode(const PlanImpl &pl, int64_t k, bool reads_inputs) {
    if (pl.rs_epilogue != 0) return pl.rs_epilogue - 1;
    if (reads_inputs) return 0;
    const int64_t kslices = (k + kBK - 1) / kBK;
    const bool many_ranks = pl.N >= 16 || (pl.N >= 8 && pl.dir == CM_RING_UNI);
    return many_ranks && kslices >= 28 ? 1 : 0;
}

// One ring stream's buckets, M*n*4 bytes, fit in L2 with room to spare up to
// this size: the automatic choices of CM_OPT_RS_IN_PLACE, CM_OPT_RS_COL_SLABS
// and CM_OPT_RS_BUCKET_HINT follow it.
constexpr int64_t kBucketsInL2Bytes = int64_t(128) << 20;

// CM_OPT_RS_BUCKET_HINT: the L2 policy of the TMA epilogue's bucket writes
// and adds (kernel: 0 none, 1 evict_first, 2 evict_last; the vector
// epilogues take none: a build whose vector epilogues also carried the
// policy variants ran the default MLP GEMM-RS 1-2 % slower).  Automatic (option 0): one
// ring stream's buckets take M*n*4 bytes; up to kBucketsInL2Bytes they can
// stay in L2 from one contribution to the next, and evict_last keeps them
// there; beyond that, no policy.  Measured (interleaved, two runs on two
// boxes, against no policy): GPT-3 attention-out (100 MB of buckets) 1.8-2.0 %
// faster one-way and 3.0-3.5 % two-way with evict_last, Megatron-SP fc2
// (67 MB) 0.6-1.5 %; on the MLP (268 MB) evict_first gained 1.8 % at N=8 in
// one run and lost 1.0-2.2 % at N=4 and 8 in the other, evict_last within
// 1 %.  Option 3: no policy.

int rs_bucket_hint(const PlanImpl &pl, int64_t M, int64_t n) {
    if (pl.rs_bucket_hint == 3) return 0;
    if (pl.rs_bucket_hint != 0) return pl.rs_bucket_hint;
    return M * n * 4 <= kBucketsInL2Bytes ? 2 : 0;
}

// CM_OPT_RS_COL_SLABS: the GEMM -> ReduceScatter tile order in that many
// passes over the tasks, one slab of column tiles each; the largest count
// not above it that divides the column tiles.  A pass touches 1/slabs of
// every bucket but reads all of X again.  Automatic (0): two slabs for a
// one-way ring whose buckets fit L2 (kBucketsInL2Bytes) and whose tiles have
// at least 16 K slices, else one pass.  Measured (interleaved, three runs):
// two slabs made the GPT-3 attention-out one-way ring 3-5 % faster (0.441
// against 0.456 ms with the bucket policy), left its two-way ring within
// 2 % (slower), and slowed the Megatron-SP fc2 (4 K slices) by 5-7 % and
// the MLP sweep (268 MB of buckets) by up to 1 %; three or more slabs were
// slower everywhere, by up to 50 %.
int rs_col_slabs(const PlanImpl &pl, int ntiles, int64_t M, int64_t n, int64_t k) {
    int c = pl.rs_col_slabs;
    if (c == 0)
        c = pl.dir == CM_RING_UNI && M * n * 4 <= kBucketsInL2Bytes && (k + kBK - 1) / kBK >= 16 ? 2 : 1;
    while (c > 1 && ntiles % c != 0) --c;
    return c;
}


// Ring stages of received bucket per tile for CM_OPT_RS_PRELOAD = mode.
int preload_stages(int mode, int64_t kslices) {
    switch (mode) {
        case 1: return 4;
        case 3: return 2;
        case 2: return kslices <= kPreloadAllKSlices ? 4 : 0;
        default: return 0;
    }
}
static_assert(kCounterOff + 4 * (CM_MAX_RANKS + 1) <= kStatusBytes, "tile counters fit the status block");

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct WsLayout {
    size_t flags_off = kStatusBytes, flags_bytes = 0, buf_off = 0, buf_bytes = 0, total = 0;
};

int streams_of(const PlanImpl &p) { return p.dir == CM_RING_BIDI ? 2 : 1; }

// Readiness counters: AG one per (flag id, chunk, row tile), RS one per (flag
// id, chunk, row tile, column tile) -- sized for the smaller (128-row) tiles
// of the two kernels, so either kernel's indices fit.
size_t row_tiles(int64_t rows_c) { return size_t((rows_c + kBM - 1) / kBM); }

WsLayout ag_layout(const PlanImpl &p, int64_t m, int64_t K) {
    WsLayout l;
    const int64_t rows_c = p.dir == CM_RING_NONE ? int64_t(p.N) * m : (m + p.chunks - 1) / p.chunks;
    l.flags_bytes = size_t(p.flag_ids[CM_OP_AG_GEMM]) * size_t(p.chunks) * row_tiles(rows_c) * sizeof(uint32_t);
    l.buf_off = align_up(l.flags_off + l.flags_bytes, 1024);
    const bool ring = p.dir != CM_RING_NONE && p.N > 1;
    const size_t slots = ring ? size_t(p.N * streams_of(p) * p.sched[CM_OP_AG_GEMM].steps) : 0;   // one per (rank, stream, step)
    l.buf_bytes = slots * size_t(m) * size_t(K) * 2;
    l.total = l.buf_off + l.buf_bytes;
    return l;
}

// CM_OPT_RS_IN_PLACE for a call of M x n: 1 in place, 0 per-step buffers, 2
// (automatic) in place where one stream's buckets fit L2, per-step buffers
// otherwise.  Measured (interleaved, each with its automatic epilogue): in
// place was 6-10 % faster on the GPT-3 attention-out (100 MB of buckets) and
// 2-3 % on the Megatron-SP fc2 (67 MB); per-step buffers were 2-4 % faster
// on the MLP at N = 4 and 8 and on the two-way N = 16 ring (268 MB), and
// even on the one-way N = 16 ring.  Where the buckets stay in L2, an add
// where the bucket lies costs one L2 read-modify-write; where they do not,
// the TMA epilogue's streaming load-add-store of per-step buffers keeps the
// tensor pipe fed better than reduce-adds that each go to DRAM.
bool rs_in_place_for(const PlanImpl &p, int64_t M, int64_t n) {
    if (p.rs_in_place != 2) return p.rs_in_place != 0;
    return M * n * 4 <= kBucketsInL2Bytes;
}

// RS accumulator buffers of [M/N][n] fp32: one per (bucket, ring stream) when
// buckets are accumulated in place, else one per (rank, ring stream, step).
int64_t rs_bufs(const PlanImpl &p, bool in_place) {
    if (p.dir == CM_RING_NONE || p.N <= 1) return 0;
    const int64_t per = in_place ? 1 : p.sched[CM_OP_GEMM_RS].steps;
    return int64_t(p.N) * streams_of(p) * per;
}

WsLayout rs_layout(const PlanImpl &p, int64_t M, int64_t n) {
    WsLayout l;
    const int64_t rows_c = (M / p.N + p.chunks - 1) / p.chunks;
    l.flags_bytes = size_t(p.flag_ids[CM_OP_GEMM_RS]) * size_t(p.chunks) * row_tiles(rows_c) *
                    size_t((n + kBN - 1) / kBN) * sizeof(uint32_t);
    l.buf_off = align_up(l.flags_off + l.flags_bytes, 1024);
    l.buf_bytes = size_t(rs_bufs(p, rs_in_place_for(p, M, n))) * size_t(M / p.N) * size_t(n) * sizeof(float);
    l.total = l.buf_off + l.buf_bytes;
    return l;
}

// Pipelined RS: the status block, then every rank's fp32 partial product of
// every bucket, [N*N][M/N][n] (buffer r*N + o).
WsLayout rs_pipe_layout(const PlanImpl &p, int64_t M, int64_t n) {
    WsLayout l;
    l.buf_off = align_up(l.flags_off, 1024);
    l.buf_bytes = size_t(p.N) * size_t(M) * size_t(n) * sizeof(float);
    l.total = l.buf_off + l.buf_bytes;
    return l;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 3-D tensor [d2][d1][d0] (d0 contiguous) of bf16 (or fp32), 128-byte swizzled boxes of b0 x b1;
// l2_promotion is the plan's CM_OPT_L2_PROMOTION (0 none, 1 64 B, 2 128 B, 3 256 B).
bool make_map(CUtensorMap *m, int l2_promotion, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
              uint32_t b1, bool f32 = false) {
    auto enc = encode_fn();
    if (!enc) return false;
    const uint64_t es_bytes = f32 ? 4 : 2;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * es_bytes, d0 * d1 * es_bytes};
    cuuint32_t box[3] = {b0, b1, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     static_cast<CUtensorMapL2promotion>(l2_promotion),
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// fp32 accumulators [slabs][rows][n] in 32 x 32 boxes (128-byte swizzle):
// the CTA-pair TMA epilogue's loads, stores and adds of bucket slices.
bool make_acc_maps(KParams &kp, int promo, const float *acc, int64_t n, int64_t rows, int64_t slabs) {
    return make_map(&kp.tmAcc, promo, acc, uint64_t(n), uint64_t(rows), uint64_t(slabs), 32, 32, true);
}

// The kernel a call runs: CTA pairs (one pair per cluster), or single CTAs.
struct KernelChoice {
    bool pair;
};

KernelChoice choose_kernel(const PlanImpl &pl) { return {pl.kernel != 1}; }

constexpr int64_t kRowBandBytes = int64_t(32) << 20;   // A bytes per row band of the tile order

// Row tiles, column tiles and flag targets for the selected kernel.
// pair_chunks: a ring call on CTA pairs of one cluster whose chunks have at
// most 128 rows puts two chunks in one 256-row pair tile, one per CTA,
// instead of leaving half of every tile on zero rows.
void set_tiling(const KernelChoice &kc, int op, KParams &kp, int64_t rows_c, int64_t n, bool pair_chunks = false) {
    const int tm = kc.pair ? pair_rows() : kBM;
    kp.chunk_pair = pair_chunks && kc.pair && kp.chunks % 2 == 0 && rows_c <= kBM;
    // signals per chunk and tile: one per CTA of a pair whose CTAs share the
    // chunk; one when each CTA of the pair has a chunk of its own
    const int per_tile = kc.pair && !kp.chunk_pair ? 2 : 1;
    kp.mtiles_c = int((rows_c + tm - 1) / tm);
    kp.ntiles = int((n + kBN - 1) / kBN);
    kp.tiles_per_task = (kp.chunk_pair ? kp.chunks / 2 : kp.chunks) * kp.mtiles_c * kp.ntiles;
    if (op == CM_OP_AG_GEMM) {
        // forwards per (chunk, row tile): CTA pairs forward a row slice from
        // every column tile (from each CTA that holds the chunk); single CTAs
        // forward the whole row tile from column tile 0
        kp.tgt_in = uint32_t(kc.pair ? per_tile * kp.ntiles : 1);
        kp.tgt_free = 0;   // receive slots are written once: nothing waits for a slot to be free
    } else {
        // signals of the same bucket tile: CTA pairs, one per warp that
        // drains it (vector epilogues: the four of a group, or all eight) or
        // one per CTA (TMA epilogue), in each CTA holding the chunk; single
        // CTAs, one per tile
        const uint32_t warps = kp.rs_epi == 1 ? kPairEpiWarps / 2 : kp.rs_epi == 2 ? kPairEpiWarps : 1;
        kp.tgt_in = uint32_t(kc.pair ? per_tile * warps : 1);
        kp.tgt_free = kp.tgt_in;
    }
}

// Launch geometry of the selected kernel for `tiles` tiles.
// layout: bit 0 = B MN-major, bit 1 = A MN-major (CTA pairs only).
cudaError_t launch_tiles(const PlanImpl &pl, const KernelChoice &kc, const KParams &kp, int layout, int64_t tiles,
                         int max_clusters, int sms, cudaStream_t stream) {
    if (kc.pair) {
        int clusters = pl.grid > 0 ? std::min(pl.grid / 2, max_clusters) : max_clusters;
        clusters = std::max(1, clusters);
        if (tiles < clusters) clusters = int(tiles);
        return launch_pair(kp, layout, clusters, stream);
    }
    if (layout & 2) return cudaErrorInvalidValue;
    int grid = pl.grid > 0 ? std::min(pl.grid, sms) : sms;
    if (tiles < grid) grid = int(tiles);
    return launch_persistent(kp, (layout & 1) != 0, grid, stream);
}

// Per-call parameters shared by every launch: status, flags, bounds, tile order.
cm_status setup_launch(const PlanImpl &pl, const KernelChoice &kc, KParams &kp, const WsLayout &l, void *ws,
                       int *sms, int *max_clusters) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CM_ERR_CUDA;
    if (prepare_device(dev, sms) != cudaSuccess) return CM_ERR_CUDA;
    *max_clusters = 0;
    if (kc.pair && prepare_pair(dev, max_clusters) != cudaSuccess) return CM_ERR_CUDA;
    if (kc.pair && *max_clusters <= 0) return CM_ERR_UNSUPPORTED;
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    kp.status = reinterpret_cast<uint32_t *>(w8);
    kp.flags = reinterpret_cast<uint32_t *>(w8 + l.flags_off);
    kp.flag_words = int64_t(l.flags_bytes / sizeof(uint32_t));
    kp.timeout_ns = uint64_t(pl.timeout_ns);
    kp.static_tiles = pl.static_tiles;
    kp.l2_hint_a = pl.l2_hints & 0xf;
    kp.l2_hint_b = (pl.l2_hints >> 4) & 0xf;
    // row bands: explicit, or as many row tiles as hold about 32 MB of A
    // (a band's A rows stay in L2 while the band runs through the columns)
    if (pl.row_band > 0) {
        kp.row_band = pl.row_band;
    } else {
        const int64_t tile_bytes = int64_t(kc.pair ? pair_rows() : kBM) * kp.kblocks * kBK * 2;
        kp.row_band = int(std::max<int64_t>(1, kRowBandBytes / tile_bytes));
    }
    return CM_OK;
}

// CM_OPT_TASK_ORDER automatic choice: a one-way ring runs step-major when the
// weight shards of all ranks together take at most this many bytes (they
// stay in L2 whichever order streams them, and step-major puts every task
// furthest from the tasks it depends on); rank-blocked otherwise (each rank's
// weight shard streamed in two runs instead of once per step).
constexpr int64_t kStepMajorWeightBytes = int64_t(48) << 20;

bool use_step_major(const PlanImpl &pl, int64_t weight_bytes) {
    if (pl.task_order == 2) return true;
    if (pl.task_order == 1) return false;
    return weight_bytes <= kStepMajorWeightBytes;
}

// rs_per_step: a GEMM -> ReduceScatter call with per-step buffers (the plan's
// second RS task table).
cm_status run(const PlanImpl &pl, const KernelChoice &kc, int op, KParams &kp, const WsLayout &l, void *ws,
              bool b_mn, bool step_major, cudaStream_t stream, bool rs_per_step = false) {
    int sms = 0, max_clusters = 0;
    cm_status st = setup_launch(pl, kc, kp, l, ws, &sms, &max_clusters);
    if (st != CM_OK) return st;
    const bool ps = op == CM_OP_GEMM_RS && rs_per_step;
    const auto &tasks = step_major ? (ps ? pl.rs_ps_sm : pl.tasks_sm[op]) : (ps ? pl.rs_ps : pl.tasks[op]);
    const int ntasks = int(tasks.size());
    if (ntasks > kMaxTasks) return CM_ERR_UNSUPPORTED;
    std::memcpy(kp.tasks, tasks.data(), sizeof(cm_task) * size_t(ntasks));
    // status word and flags start at zero for every call
    if (cudaMemsetAsync(ws, 0, l.buf_off, stream) != cudaSuccess) return CM_ERR_CUDA;
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    const auto &sb = step_major ? (ps ? pl.rs_ps_step_begin_sm : pl.step_begin_sm[op])
                                : (ps ? pl.rs_ps_step_begin : pl.step_begin[op]);
    const int nsteps = int(sb.size()) - 1;
    const int launches = pl.serial_steps ? nsteps : 1;
    for (int i = 0; i < launches; ++i) {
        // each launch has its own tile counter (zeroed with the flags)
        kp.tile_counter = reinterpret_cast<uint32_t *>(w8 + kCounterOff) + i;
        kp.task_begin = pl.serial_steps ? sb[size_t(i)] : 0;
        kp.task_end = pl.serial_steps ? sb[size_t(i) + 1] : ntasks;
        if (kp.task_end <= kp.task_begin) continue;
        const int64_t tiles = int64_t(kp.task_end - kp.task_begin) * kp.tiles_per_task;
        if (launch_tiles(pl, kc, kp, b_mn ? 1 : 0, tiles, max_clusters, sms, stream) != cudaSuccess)
            return CM_ERR_CUDA;
    }
    return CM_OK;
}

// The library's second stream per device (non-blocking) and its events: the
// pipelined RS runs each chunk's reduction there, ordered after that chunk's
// GEMM by an event; the caller's stream waits for the last reduction.
constexpr int kMaxDevices = 64;
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t ev[CM_MAX_CHUNKS + 1] = {};
};

enum SideUser { kSidePipelinedRs = 0, kSideBackwardPair = 1, kSideCannon = 2 };

SideStream *side_stream(int dev, SideUser user) {   // caller holds that user's call mutex
    static SideStream ss[3][kMaxDevices];
    SideStream &d = ss[user][dev];
    if (!d.stream) {
        if (cudaStreamCreateWithFlags(&d.stream, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        for (auto &e : d.ev)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    }
    return &d;
}

cm_status check_common(cm_plan_t plan, const void *x, const void *w, cm_wlayout wl, void *y, cm_dtype yd,
                       int64_t rows, int64_t K, int64_t n) {
    if (!plan || !x || !w || !y) return CM_ERR_INVALID_ARG;
    if (wl != CM_W_KN && wl != CM_W_NK) return CM_ERR_INVALID_ARG;
    if (yd != CM_BF16 && yd != CM_F32) return CM_ERR_INVALID_ARG;
    if (rows <= 0 || K <= 0 || n <= 0) return CM_ERR_SHAPE;
    if (K % 8 != 0 || n % 8 != 0) return CM_ERR_ALIGNMENT;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return CM_ERR_ALIGNMENT;
    if (K > (int64_t(1) << 30) || n > (int64_t(1) << 30) || rows > (int64_t(1) << 30)) return CM_ERR_SHAPE;
    return CM_OK;
}

}  // namespace
}  // namespace cm

using namespace cm;

// An NVTX range for the host side of one call (and of each step a call
// enqueues): profilers show which call a launch belongs to, and ncu can be
// limited to one call with --nvtx --nvtx-include.  With no tool attached a
// range costs a branch.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

extern "C" {

size_t cm_ag_gemm_workspace_size(cm_plan_t plan, int64_t m, int64_t K) {
    if (!plan || m <= 0 || K <= 0) return 0;
    return ag_layout(plan->impl, m, K).total;
}

size_t cm_gemm_rs_workspace_size(cm_plan_t plan, int64_t M, int64_t n) {
    if (!plan || M <= 0 || n <= 0) return 0;
    return rs_layout(plan->impl, M, n).total;
}

cm_status cm_ag_gemm(cm_plan_t plan, const void *x, const void *w, cm_wlayout wlayout, void *y, cm_dtype y_dtype,
                     int64_t m, int64_t K, int64_t n, void *ws, size_t ws_bytes, cm_stream_t stream) {
    const NvtxRange range("cm_ag_gemm");
    cm_status st = check_common(plan, x, w, wlayout, y, y_dtype, m, K, n);
    if (st != CM_OK) return st;
    const PlanImpl &pl = plan->impl;
    const int N = pl.N;
    if (m % pl.chunks != 0) return CM_ERR_SHAPE;
    const WsLayout l = ag_layout(pl, m, K);
    if (!ws || ws_bytes < l.total) return CM_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return CM_ERR_ALIGNMENT;

    const bool none = pl.dir == CM_RING_NONE;
    const int c = none ? 1 : pl.chunks;
    const int64_t rows_c = none ? int64_t(N) * m : m / c;
    const int64_t slabs = none ? 1 : int64_t(N) * c;
    static KParams kp;   // ~9 KB; calls are serialised by the mutex below
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    std::memset(static_cast<void *>(&kp), 0, sizeof kp);
    kp.q_only = -1;
    const int promo = pl.l2_promotion;
    const KernelChoice kc = choose_kernel(pl);
    // A box: a CTA's 128 rows (fewer when a chunk is shorter)
    const uint32_t box_rows = uint32_t(std::min<int64_t>(kBM, rows_c));
    if (!make_map(&kp.tmA0, promo, x, uint64_t(K), uint64_t(rows_c), uint64_t(slabs), kBK, box_rows)) return CM_ERR_CUDA;
    uint8_t *bufs = static_cast<uint8_t *>(ws) + l.buf_off;
    if (l.buf_bytes > 0) {
        const int64_t nslots = int64_t(N) * streams_of(pl) * pl.sched[CM_OP_AG_GEMM].steps;
        if (!make_map(&kp.tmA1, promo, bufs, uint64_t(K), uint64_t(rows_c), uint64_t(nslots * c), kBK, box_rows))
            return CM_ERR_CUDA;
    } else {
        kp.tmA1 = kp.tmA0;
    }
    const bool b_mn = wlayout == CM_W_KN;
    const uint32_t b_rows = kc.pair ? kBN / 2 : kBN;   // a pair CTA stages half the columns
    if (b_mn) {
        if (!make_map(&kp.tmB, promo, w, uint64_t(n), uint64_t(K), uint64_t(N), 64, kBK)) return CM_ERR_CUDA;
    } else {
        if (!make_map(&kp.tmB, promo, w, uint64_t(K), uint64_t(n), uint64_t(N), kBK, b_rows)) return CM_ERR_CUDA;
    }
    kp.y = y;
    kp.acc = nullptr;
    kp.x_bytes = static_cast<const uint8_t *>(x);
    kp.slot_bytes = bufs;
    kp.x_total = int64_t(N) * m * K * 2;
    kp.slot_total = int64_t(l.buf_bytes);
    kp.y_elems = int64_t(N) * N * m * n;
    kp.a0_slabs = int(slabs);
    kp.a1_slabs = l.buf_bytes > 0 ? int(int64_t(N) * streams_of(pl) * pl.sched[CM_OP_AG_GEMM].steps * c) : int(slabs);
    kp.b_slabs = N;
    kp.row_bytes = K * 2;
    kp.y_rank_stride = int64_t(N) * m * n;
    kp.out_rows_per_idx = none ? int64_t(N) * m : m;
    kp.acc_buf_stride = 0;
    kp.op = 0;
    kp.N = N;
    kp.chunks = c;
    kp.rows_c = int(rows_c);
    kp.kblocks = int((K + kBK - 1) / kBK);
    kp.n = int(n);
    kp.y_f32 = y_dtype == CM_F32;
    kp.a_box_rows = int(box_rows);
    set_tiling(kc, CM_OP_AG_GEMM, kp, rows_c, n, true);
    const bool sm = use_step_major(pl, int64_t(N) * K * n * 2);
    return run(pl, kc, CM_OP_AG_GEMM, kp, l, ws, b_mn, sm, reinterpret_cast<cudaStream_t>(stream));
}

cm_status cm_gemm_rs(cm_plan_t plan, const void *x, const void *w, cm_wlayout wlayout, void *y, cm_dtype y_dtype,
                     int64_t M, int64_t k, int64_t n, void *ws, size_t ws_bytes, cm_stream_t stream) {
    const NvtxRange range("cm_gemm_rs");
    cm_status st = check_common(plan, x, w, wlayout, y, y_dtype, M, k, n);
    if (st != CM_OK) return st;
    const PlanImpl &pl = plan->impl;
    const int N = pl.N;
    if (M % N != 0) return CM_ERR_SHAPE;
    const int64_t Mb = M / N;
    if (Mb % pl.chunks != 0) return CM_ERR_SHAPE;
    const WsLayout l = rs_layout(pl, M, n);
    if (!ws || ws_bytes < l.total) return CM_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return CM_ERR_ALIGNMENT;

    const bool none = pl.dir == CM_RING_NONE;
    const int c = none ? 1 : pl.chunks;
    const int64_t rows_c = Mb / c;
    static KParams kp;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    std::memset(static_cast<void *>(&kp), 0, sizeof kp);
    kp.q_only = -1;
    const int promo = pl.l2_promotion;
    const KernelChoice kc = choose_kernel(pl);
    const uint32_t box_rows = uint32_t(std::min<int64_t>(kBM, rows_c));
    // x [N][M][k] viewed as [N*N*c][rows_c][k]: slab (r*N + bucket)*c + chunk
    if (!make_map(&kp.tmA0, promo, x, uint64_t(k), uint64_t(rows_c), uint64_t(N) * N * c, kBK, box_rows)) return CM_ERR_CUDA;
    kp.tmA1 = kp.tmA0;
    const bool b_mn = wlayout == CM_W_KN;
    const uint32_t b_rows = kc.pair ? kBN / 2 : kBN;
    if (b_mn) {
        if (!make_map(&kp.tmB, promo, w, uint64_t(n), uint64_t(k), uint64_t(N), 64, kBK)) return CM_ERR_CUDA;
    } else {
        if (!make_map(&kp.tmB, promo, w, uint64_t(k), uint64_t(n), uint64_t(N), kBK, b_rows)) return CM_ERR_CUDA;
    }
    kp.y = y;
    kp.acc = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + l.buf_off);
    kp.y_elems = M * n;
    const bool in_place = rs_in_place_for(pl, M, n);
    kp.acc_bufs = int(rs_bufs(pl, in_place));
    kp.a0_slabs = kp.a1_slabs = N * N * c;
    kp.b_slabs = N;
    kp.bucket_hint = rs_bucket_hint(pl, M, n);
    if (l.buf_bytes > 0) {   // accumulators as [bufs*chunks][rows_c][n] fp32, 32 x 32 boxes
        const int64_t nbufs = rs_bufs(pl, in_place);
        if (!make_acc_maps(kp, promo, kp.acc, n, rows_c, nbufs * c)) return CM_ERR_CUDA;
        // received buckets through the operand ring: each CTA of a pair loads
        // its 128 rows of the tile as 32-column boxes (one per 16 KB stage
        // half); with buckets kept in place only the owner's tiles read one
        const int pre_stages = preload_stages(pl.rs_preload, (k + kBK - 1) / kBK);
        if (pre_stages > 0 && kc.pair) {
            const uint32_t pre_rows = uint32_t(std::min<int64_t>(kBM, rows_c));
            if (!make_map(&kp.tmAccIn, promo, kp.acc, uint64_t(n), uint64_t(rows_c), uint64_t(nbufs * c), 32, pre_rows, true))
                return CM_ERR_CUDA;
            kp.rs_preload = 1;
            kp.pre_stages = pre_stages;
            kp.pre_box_rows = int(pre_rows);
        }
    }
    kp.y_rank_stride = 0;
    kp.out_rows_per_idx = Mb;
    kp.acc_buf_stride = Mb * n;
    kp.op = 1;
    kp.N = N;
    kp.chunks = c;
    kp.rows_c = int(rows_c);
    kp.kblocks = int((k + kBK - 1) / kBK);
    kp.n = int(n);
    kp.y_f32 = y_dtype == CM_F32;
    kp.a_box_rows = int(box_rows);
    kp.rs_epi = rs_epi_mode(pl, k, !in_place);
    set_tiling(kc, CM_OP_GEMM_RS, kp, rows_c, n, true);
    kp.col_slabs = rs_col_slabs(pl, kp.ntiles, M, n, k);
    const bool sm = use_step_major(pl, int64_t(N) * k * n * 2);
    return run(pl, kc, CM_OP_GEMM_RS, kp, l, ws, b_mn, sm, reinterpret_cast<cudaStream_t>(stream), !in_place);
}

size_t cm_gemm_rs_pipelined_workspace_size(cm_plan_t plan, int64_t M, int64_t n) {
    if (!plan || M <= 0 || n <= 0) return 0;
    return rs_pipe_layout(plan->impl, M, n).total;
}

cm_status cm_gemm_rs_pipelined(cm_plan_t plan, const void *x, const void *w, cm_wlayout wlayout, void *y,
                               cm_dtype y_dtype, int64_t M, int64_t k, int64_t n, void *ws, size_t ws_bytes,
                               cm_stream_t stream) {
    const NvtxRange range("cm_gemm_rs_pipelined");
    cm_status st = check_common(plan, x, w, wlayout, y, y_dtype, M, k, n);
    if (st != CM_OK) return st;
    const PlanImpl &pl = plan->impl;
    const int N = pl.N;
    if (M % N != 0) return CM_ERR_SHAPE;
    const int64_t Mb = M / N;
    const int c = pl.chunks;
    if (Mb % c != 0) return CM_ERR_SHAPE;
    const WsLayout l = rs_pipe_layout(pl, M, n);
    if (!ws || ws_bytes < l.total) return CM_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return CM_ERR_ALIGNMENT;
    const int64_t rows_c = Mb / c;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    static KParams kp;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CM_ERR_CUDA;
    SideStream *ss = side_stream(dev, kSidePipelinedRs);
    if (!ss) return CM_ERR_CUDA;
    std::memset(static_cast<void *>(&kp), 0, sizeof kp);
    const int promo = pl.l2_promotion;
    const KernelChoice kc = choose_kernel(pl);
    const uint32_t box_rows = uint32_t(std::min<int64_t>(kBM, rows_c));
    // x [N][M][k] viewed as [N*N*c][rows_c][k]: slab (r*N + bucket)*c + chunk
    if (!make_map(&kp.tmA0, promo, x, uint64_t(k), uint64_t(rows_c), uint64_t(N) * N * c, kBK, box_rows)) return CM_ERR_CUDA;
    kp.tmA1 = kp.tmA0;
    const bool b_mn = wlayout == CM_W_KN;
    const uint32_t b_rows = kc.pair ? kBN / 2 : kBN;
    if (b_mn) {
        if (!make_map(&kp.tmB, promo, w, uint64_t(n), uint64_t(k), uint64_t(N), 64, kBK)) return CM_ERR_CUDA;
    } else {
        if (!make_map(&kp.tmB, promo, w, uint64_t(k), uint64_t(n), uint64_t(N), kBK, b_rows)) return CM_ERR_CUDA;
    }
    // partial products as [N*N*c][rows_c][n] fp32: slab (r*N + bucket)*c + chunk
    float *P = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + l.buf_off);
    if (!make_acc_maps(kp, promo, P, n, rows_c, int64_t(N) * N * c)) return CM_ERR_CUDA;
    kp.y = y;
    kp.acc = P;
    kp.y_elems = M * n;
    kp.acc_bufs = N * N;
    kp.a0_slabs = kp.a1_slabs = N * N * c;
    kp.b_slabs = N;
    kp.y_rank_stride = 0;
    kp.out_rows_per_idx = Mb;
    kp.acc_buf_stride = Mb * n;
    kp.op = 1;
    kp.N = N;
    kp.chunks = c;
    kp.rows_c = int(rows_c);
    kp.kblocks = int((k + kBK - 1) / kBK);
    kp.n = int(n);
    kp.y_f32 = y_dtype == CM_F32;
    kp.a_box_rows = int(box_rows);
    kp.rs_epi = rs_epi_mode(pl, k, false);
    // chunks of at most 128 rows go two to a launch, one per CTA of each pair
    // tile (the ring path's chunk pairing), instead of half-empty pair tiles
    set_tiling(kc, CM_OP_GEMM_RS, kp, rows_c, n, true);
    kp.tiles_per_task = kp.mtiles_c * kp.ntiles;   // one chunk (or chunk pair) per launch
    const int per_launch = kp.chunk_pair ? 2 : 1;
    kp.tgt_in = kp.tgt_free = 0;
    int sms = 0, max_clusters = 0;
    st = setup_launch(pl, kc, kp, l, ws, &sms, &max_clusters);
    if (st != CM_OK) return st;
    // one task per (rank r, bucket o): X_r's rows of bucket o times W_r, stored
    // as an fp32 partial; no ring, no flags
    const int ntasks = N * N;
    if (ntasks > kMaxTasks) return CM_ERR_UNSUPPORTED;
    for (int r = 0; r < N; ++r)
        for (int o = 0; o < N; ++o) {
            cm_task &t = kp.tasks[r * N + o];
            std::memset(&t, 0xff, sizeof t);   // every field -1 ...
            t.rank = int16_t(r);
            t.a_slab = int16_t(r * N + o);
            t.a_src = 0;
            t.out_idx = int16_t(o);
            t.out_buf = int16_t(r * N + o);
            t.step = 0;
            t.stream = 0;
            const int g = std::max(1, std::min(pl.tile_group, N));   // runs of one rank's buckets
            const int first = (o / g) * g, size = std::min(g, N - first);
            t.tile_group = int16_t((size << 8) | (o - first));
        }
    kp.task_begin = 0;
    kp.task_end = ntasks;
    if (cudaMemsetAsync(ws, 0, l.buf_off, s) != cudaSuccess) return CM_ERR_CUDA;
    for (int g = 0; g < c / per_launch; ++g) {
        // GEMM of chunk g (or chunks 2g and 2g + 1) on the caller's stream;
        // their reduction on the side stream, under the next launch's GEMM
        kp.q_only = g;
        kp.tile_counter = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) + kCounterOff) + g;
        const int64_t tiles = int64_t(ntasks) * kp.tiles_per_task;
        if (launch_tiles(pl, kc, kp, b_mn ? 1 : 0, tiles, max_clusters, sms, s) != cudaSuccess) return CM_ERR_CUDA;
        if (cudaEventRecord(ss->ev[g], s) != cudaSuccess) return CM_ERR_CUDA;
        if (cudaStreamWaitEvent(ss->stream, ss->ev[g], 0) != cudaSuccess) return CM_ERR_CUDA;
        for (int j = g * per_launch; j < (g + 1) * per_launch; ++j)
            if (launch_reduce_chunk(P, y, N, Mb, rows_c, n, j, y_dtype == CM_F32, sms, ss->stream) != cudaSuccess)
                return CM_ERR_CUDA;
    }
    if (cudaEventRecord(ss->ev[CM_MAX_CHUNKS], ss->stream) != cudaSuccess) return CM_ERR_CUDA;
    if (cudaStreamWaitEvent(s, ss->ev[CM_MAX_CHUNKS], 0) != cudaSuccess) return CM_ERR_CUDA;
    return CM_OK;
}

// Backward pair workspace: the data gradient's GEMM-RS workspace, a status
// block for the weight-gradient launch, then every rank's gathered input.
struct BwdLayout {
    size_t rs_bytes = 0, wg_off = 0, xg_off = 0, total = 0;
};

BwdLayout bwd_layout(const PlanImpl &p, int64_t m, int64_t K, int64_t n) {
    (void)n;
    BwdLayout b;
    b.rs_bytes = rs_layout(p, int64_t(p.N) * m, K).total;
    b.wg_off = align_up(b.rs_bytes, 1024);
    b.xg_off = b.wg_off + 1024;
    b.total = b.xg_off + size_t(p.N) * size_t(p.N) * size_t(m) * size_t(K) * 2;
    return b;
}

size_t cm_backward_pair_workspace_size(cm_plan_t plan, int64_t m, int64_t K, int64_t n) {
    if (!plan || m <= 0 || K <= 0 || n <= 0) return 0;
    return bwd_layout(plan->impl, m, K, n).total;
}

cm_status cm_backward_pair(cm_plan_t plan, const void *x, const void *w, const void *dy, void *dx, cm_dtype dx_dtype,
                           void *dw, cm_dtype dw_dtype, int64_t m, int64_t K, int64_t n, void *ws, size_t ws_bytes,
                           cm_stream_t stream) {
    const NvtxRange range("cm_backward_pair");
    if (!plan || !x || !w || !dy || !dx || !dw) return CM_ERR_INVALID_ARG;
    if ((dx_dtype != CM_BF16 && dx_dtype != CM_F32) || (dw_dtype != CM_BF16 && dw_dtype != CM_F32))
        return CM_ERR_INVALID_ARG;
    const PlanImpl &pl = plan->impl;
    const int N = pl.N;
    const int64_t T = int64_t(N) * m;   // tokens: the gathered rows
    if (m <= 0 || K <= 0 || n <= 0) return CM_ERR_SHAPE;
    if (K % 8 != 0 || n % 8 != 0) return CM_ERR_ALIGNMENT;
    if (n < 64 || K < 64 || T < 64 || m % pl.chunks != 0) return CM_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(w) || !aligned16(dy) || !aligned16(dx) || !aligned16(dw)) return CM_ERR_ALIGNMENT;
    const BwdLayout bl = bwd_layout(pl, m, K, n);
    if (!ws || ws_bytes < bl.total) return CM_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return CM_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    uint8_t *xg = w8 + bl.xg_off;   // [N ranks][T][K] bf16

    static KParams kp;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CM_ERR_CUDA;
    SideStream *ss = side_stream(dev, kSideBackwardPair);
    if (!ss) return CM_ERR_CUDA;

    // 1. the weight gradient's AllGather: every rank's copy of concat_j(X_j),
    //    on the second stream (after the work already queued on `stream`)
    const size_t shard = size_t(m) * size_t(K) * 2;
    cudaStream_t ag = pl.bulk_overlap ? ss->stream : s;
    if (pl.bulk_overlap) {
        if (cudaEventRecord(ss->ev[0], s) != cudaSuccess) return CM_ERR_CUDA;
        if (cudaStreamWaitEvent(ag, ss->ev[0], 0) != cudaSuccess) return CM_ERR_CUDA;
    }
    // rank r receives shards 0..N-1 in order, into one contiguous [T][K]
    // buffer: shard j of x lands at row block j, so the N shards of one rank
    // go as one copy (fewer, larger copies keep the copy engine's per-copy
    // cost off the critical path)
    for (int r = 0; r < N; ++r)
        if (cudaMemcpyAsync(xg + size_t(r) * N * shard, x, size_t(N) * shard, cudaMemcpyDeviceToDevice, ag) !=
            cudaSuccess)
            return CM_ERR_CUDA;
    if (pl.bulk_overlap && cudaEventRecord(ss->ev[1], ag) != cudaSuccess) return CM_ERR_CUDA;

    // 2. the data gradient: GEMM -> ReduceScatter of dY_r @ W_r on the ring
    cm_status st = cm_gemm_rs(plan, dy, w, CM_W_KN, dx, dx_dtype, T, n, K, ws, bl.rs_bytes, stream);
    if (st != CM_OK) return st;

    // 3. the weight gradient once the gather has landed: one GEMM per rank,
    //    A = dY_r^T (MN-major) and B = the rank's gathered input (MN-major)
    if (pl.bulk_overlap && cudaStreamWaitEvent(s, ss->ev[1], 0) != cudaSuccess) return CM_ERR_CUDA;
    std::memset(static_cast<void *>(&kp), 0, sizeof kp);
    kp.q_only = -1;
    const int promo = pl.l2_promotion;
    KernelChoice kc;
    kc.pair = true;
    if (!make_map(&kp.tmA0, promo, dy, uint64_t(n), uint64_t(T), uint64_t(N), 64, kBK)) return CM_ERR_CUDA;
    kp.tmA1 = kp.tmA0;
    if (!make_map(&kp.tmB, promo, xg, uint64_t(K), uint64_t(T), uint64_t(N), 64, kBK)) return CM_ERR_CUDA;
    kp.y = dw;
    kp.y_elems = int64_t(N) * n * K;
    kp.a0_slabs = kp.a1_slabs = kp.b_slabs = N;
    kp.y_rank_stride = n * K;
    kp.out_rows_per_idx = n;
    kp.op = 0;
    kp.N = N;
    kp.chunks = 1;
    kp.rows_c = int(n);
    kp.kblocks = int((T + kBK - 1) / kBK);
    kp.n = int(K);
    kp.y_f32 = dw_dtype == CM_F32;
    kp.a_box_rows = kBM;   // an MN-major half is always two full 64-wide boxes
    set_tiling(kc, CM_OP_AG_GEMM, kp, n, K);
    kp.tgt_in = kp.tgt_free = 0;
    for (int r = 0; r < N; ++r) {
        cm_task &t = kp.tasks[r];
        std::memset(&t, 0xff, sizeof t);   // every field -1 ...
        t.rank = int16_t(r);
        t.a_slab = int16_t(r);
        t.a_src = 0;
        t.out_idx = 0;
        t.step = 0;
        t.stream = 0;
        t.tile_group = int16_t(1 << 8);
    }
    kp.task_begin = 0;
    kp.task_end = N;
    WsLayout l;   // the weight-gradient launch's own status block and counters
    l.flags_off = 0;
    l.buf_off = 256;
    int sms = 0, max_clusters = 0;
    st = setup_launch(pl, kc, kp, l, w8 + bl.wg_off, &sms, &max_clusters);
    if (st != CM_OK) return st;
    // failures go to the call's status word (cleared by the GEMM-RS above),
    // so cm_check_status(ws) covers both launches; the tile counter is fresh
    kp.status = reinterpret_cast<uint32_t *>(w8);
    kp.tile_counter = reinterpret_cast<uint32_t *>(w8 + bl.wg_off + kCounterOff);
    if (cudaMemsetAsync(w8 + bl.wg_off, 0, 256, s) != cudaSuccess) return CM_ERR_CUDA;
    if (launch_tiles(pl, kc, kp, 3, int64_t(N) * kp.tiles_per_task, max_clusters, sms, s) != cudaSuccess)
        return CM_ERR_CUDA;
    return CM_OK;
}

// Device-to-device copies issued in order, with each copy that continues the
// previous one in both source and destination merged into it: a rotation
// by whole blocks becomes a few large copies instead of one per block.
struct CopyList {
    struct C {
        uint8_t *dst;
        const uint8_t *src;
        size_t bytes;
    };
    C c[2 * CM_MAX_RANKS];
    int n = 0;
    void add(uint8_t *dst, const uint8_t *src, size_t bytes) {
        if (n > 0 && c[n - 1].dst + c[n - 1].bytes == dst && c[n - 1].src + c[n - 1].bytes == src) {
            c[n - 1].bytes += bytes;
            return;
        }
        c[n++] = C{dst, src, bytes};
    }
    bool issue(cudaStream_t st) const {
        for (int k = 0; k < n; ++k)
            if (cudaMemcpyAsync(c[k].dst, c[k].src, c[k].bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
                return false;
        return true;
    }
};

// Cannon workspace: the status block, two fp32 accumulators per rank
// (ping-pong across steps), then two sets of rotated A blocks and two of B.
struct CannonLayout {
    size_t acc_off = 0, a_off = 0, b_off = 0, total = 0;
};

CannonLayout cannon_layout(int P, int64_t bm, int64_t bk, int64_t bn) {
    CannonLayout c;
    c.acc_off = 1024;
    c.a_off = align_up(c.acc_off + size_t(P) * 2 * size_t(bm) * size_t(bn) * 4, 1024);
    c.b_off = align_up(c.a_off + 2 * size_t(P) * size_t(bm) * size_t(bk) * 2, 1024);
    c.total = c.b_off + 2 * size_t(P) * size_t(bk) * size_t(bn) * 2;
    return c;
}

int grid_side(int P) {   // q with q * q == P, else 0
    for (int q = 1; q * q <= P; ++q)
        if (q * q == P) return q;
    return 0;
}

size_t cm_cannon_workspace_size(cm_plan_t plan, int64_t bm, int64_t bk, int64_t bn) {
    if (!plan || bm <= 0 || bk <= 0 || bn <= 0 || grid_side(plan->impl.N) == 0) return 0;
    return cannon_layout(plan->impl.N, bm, bk, bn).total;
}

cm_status cm_cannon_gemm(cm_plan_t plan, const void *a, const void *b, cm_wlayout blayout, void *c, cm_dtype c_dtype,
                         int64_t bm, int64_t bk, int64_t bn, void *ws, size_t ws_bytes, cm_stream_t stream) {
    const NvtxRange range("cm_cannon_gemm");
    cm_status st = check_common(plan, a, b, blayout, c, c_dtype, bm, bk, bn);
    if (st != CM_OK) return st;
    const PlanImpl &pl = plan->impl;
    const int P = pl.N, q = grid_side(P);
    if (q == 0) return CM_ERR_SHAPE;
    const CannonLayout cl = cannon_layout(P, bm, bk, bn);
    if (!ws || ws_bytes < cl.total) return CM_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return CM_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    float *acc = reinterpret_cast<float *>(w8 + cl.acc_off);
    const size_t a_blk = size_t(bm) * size_t(bk) * 2, b_blk = size_t(bk) * size_t(bn) * 2;
    uint8_t *aset[2] = {w8 + cl.a_off, w8 + cl.a_off + size_t(P) * a_blk};
    uint8_t *bset[2] = {w8 + cl.b_off, w8 + cl.b_off + size_t(P) * b_blk};
    const uint8_t *a_in = static_cast<const uint8_t *>(a), *b_in = static_cast<const uint8_t *>(b);

    static KParams kp;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CM_ERR_CUDA;
    SideStream *ss = side_stream(dev, kSideCannon);
    if (!ss) return CM_ERR_CUDA;
    // events: ev[0] start, ev[1 + s] rotation into step s ready (s >= 1),
    // ev[1 + q + s] GEMM of step s done -- 1 + 2q <= CM_MAX_CHUNKS + 1 for q <= 4
    cudaEvent_t *ev = ss->ev;
    std::memset(static_cast<void *>(&kp), 0, sizeof kp);
    kp.q_only = -1;
    const int promo = pl.l2_promotion;
    const KernelChoice kc = choose_kernel(pl);
    const bool b_mn = blayout == CM_W_KN;
    const uint32_t box_rows = uint32_t(std::min<int64_t>(kBM, bm));
    if (!make_acc_maps(kp, promo, acc, bn, bm, int64_t(P) * 2)) return CM_ERR_CUDA;
    kp.y = c;
    kp.acc = acc;
    kp.y_elems = int64_t(P) * bm * bn;
    kp.acc_bufs = P * 2;
    kp.a0_slabs = kp.a1_slabs = kp.b_slabs = P;
    kp.out_rows_per_idx = bm;
    kp.acc_buf_stride = bm * bn;
    kp.op = 1;
    kp.N = P;
    kp.chunks = 1;
    kp.rows_c = int(bm);
    kp.kblocks = int((bk + kBK - 1) / kBK);
    kp.n = int(bn);
    kp.y_f32 = c_dtype == CM_F32;
    kp.a_box_rows = int(box_rows);
    kp.rs_epi = rs_epi_mode(pl, bk, true);
    set_tiling(kc, CM_OP_GEMM_RS, kp, bm, bn);
    kp.tgt_in = kp.tgt_free = 0;
    WsLayout l;
    l.flags_off = 256;
    l.buf_off = 1024;
    int sms = 0, max_clusters = 0;
    st = setup_launch(pl, kc, kp, l, ws, &sms, &max_clusters);
    if (st != CM_OK) return st;
    if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) return CM_ERR_CUDA;
    if (cudaEventRecord(ev[0], s) != cudaSuccess) return CM_ERR_CUDA;
    auto held_k = [q](int i, int j, int step) { return (i + j + step) % q; };
    for (int step = 0; step < q; ++step) {
        const NvtxRange step_range("cm_cannon_gemm step");
        // GEMM of this step: rank (i, j) multiplies A_{i,k} B_{k,j}, k = (i+j+step) mod q,
        // adding the accumulator of the previous step; the last step writes C
        if (step > 0 && cudaStreamWaitEvent(s, ev[1 + step], 0) != cudaSuccess) return CM_ERR_CUDA;
        const void *asrc = step == 0 ? static_cast<const void *>(a_in) : aset[step % 2];
        const void *bsrc = step == 0 ? static_cast<const void *>(b_in) : bset[step % 2];
        if (!make_map(&kp.tmA0, promo, asrc, uint64_t(bk), uint64_t(bm), uint64_t(P), kBK, box_rows)) return CM_ERR_CUDA;
        kp.tmA1 = kp.tmA0;
        if (b_mn) {
            if (!make_map(&kp.tmB, promo, bsrc, uint64_t(bn), uint64_t(bk), uint64_t(P), 64, kBK)) return CM_ERR_CUDA;
        } else {
            const uint32_t b_rows = kc.pair ? kBN / 2 : kBN;
            if (!make_map(&kp.tmB, promo, bsrc, uint64_t(bk), uint64_t(bn), uint64_t(P), kBK, b_rows)) return CM_ERR_CUDA;
        }
        for (int rho = 0; rho < P; ++rho) {
            const int i = rho / q, j = rho % q, k = held_k(i, j, 0);
            cm_task &t = kp.tasks[rho];
            std::memset(&t, 0xff, sizeof t);   // every field -1 ...
            t.a_src = 0;
            t.a_slab = int16_t(step == 0 ? i * q + k : rho);    // skewed input block, or the rotated one
            t.rank = int16_t(step == 0 ? k * q + j : rho);      // B slab
            t.out_idx = int16_t(rho);
            t.in_buf[0] = int16_t(step > 0 ? rho * 2 + (step - 1) % 2 : -1);
            t.out_buf = int16_t(step + 1 < q ? rho * 2 + step % 2 : -1);
            t.step = int16_t(step);
            t.stream = 0;
            t.tile_group = int16_t(1 << 8);
        }
        kp.task_begin = 0;
        kp.task_end = P;
        kp.tile_counter = reinterpret_cast<uint32_t *>(w8 + kCounterOff) + step;
        if (launch_tiles(pl, kc, kp, b_mn ? 1 : 0, int64_t(P) * kp.tiles_per_task, max_clusters, sms, s) !=
            cudaSuccess)
            return CM_ERR_CUDA;
        if (cudaEventRecord(ev[1 + q + step], s) != cudaSuccess) return CM_ERR_CUDA;
        // rotation into step + 1 on the second stream, under this GEMM: rank
        // (i, j) receives A from (i, j+1) and B from (i+1, j).  It writes the
        // set the GEMM of step - 1 read, so it waits for that GEMM.
        if (step + 1 < q) {
            const int nx = step + 1;
            if (step == 0 && cudaStreamWaitEvent(ss->stream, ev[0], 0) != cudaSuccess) return CM_ERR_CUDA;
            if (step >= 1 && cudaStreamWaitEvent(ss->stream, ev[1 + q + step - 1], 0) != cudaSuccess)
                return CM_ERR_CUDA;
            CopyList cl;
            for (int rho = 0; rho < P; ++rho) {
                const int i = rho / q, j = rho % q;
                const int ra = i * q + (j + 1) % q;   // right neighbour
                cl.add(aset[nx % 2] + size_t(rho) * a_blk,
                       step == 0 ? a_in + size_t(i * q + held_k(i, (j + 1) % q, 0)) * a_blk
                                 : aset[step % 2] + size_t(ra) * a_blk,
                       a_blk);
            }
            for (int rho = 0; rho < P; ++rho) {
                const int i = rho / q, j = rho % q;
                const int rb = ((i + 1) % q) * q + j;   // lower neighbour
                cl.add(bset[nx % 2] + size_t(rho) * b_blk,
                       step == 0 ? b_in + size_t(held_k((i + 1) % q, j, 0) * q + j) * b_blk
                                 : bset[step % 2] + size_t(rb) * b_blk,
                       b_blk);
            }
            if (!cl.issue(ss->stream)) return CM_ERR_CUDA;
            if (cudaEventRecord(ev[1 + nx], ss->stream) != cudaSuccess) return CM_ERR_CUDA;
        }
    }
    return CM_OK;
}

cm_status cm_check_status(const void *ws, cm_stream_t stream, int32_t info[4]) {
    if (!ws) return CM_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return CM_ERR_CUDA;
    uint32_t h[4] = {0, 0, 0, 0};
    if (cudaMemcpy(h, ws, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return CM_ERR_CUDA;
    if (info)
        for (int i = 0; i < 4; ++i) info[i] = int32_t(h[i]);
    if (h[0] == 0) return CM_OK;
    if (h[0] == uint32_t(CM_ERR_TIMEOUT) || h[0] == uint32_t(CM_ERR_BOUNDS)) return cm_status(h[0]);
    return CM_ERR_CUDA;
}

const char *cm_status_string(cm_status s) {
    switch (s) {
        case CM_OK: return "ok";
        case CM_ERR_INVALID_ARG: return "invalid argument";
        case CM_ERR_SHAPE: return "shape not supported (divisibility)";
        case CM_ERR_ALIGNMENT: return "pointer or extent not aligned for TMA";
        case CM_ERR_UNSUPPORTED: return "unsupported configuration";
        case CM_ERR_CUDA: return "CUDA error";
        case CM_ERR_TIMEOUT: return "device-side wait timed out";
        case CM_ERR_WORKSPACE: return "workspace missing or too small";
        case CM_ERR_BOUNDS: return "computed index outside its buffer (bounds-checked build)";
    }
    return "unknown status";
}

#ifdef CM_DEBUG_BOUNDS
const char *cm_version(void) { return "cm 0.2 (sm_103a tcgen05/TMA persistent kernel; bounds-checked)"; }
#else
const char *cm_version(void) { return "cm 0.2 (sm_103a tcgen05/TMA persistent kernel)"; }
#endif

}  // extern "C"
