// cm_kernel.cuh -- parameters and launch entry of the persistent tile kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "cm_internal.h"

namespace cm {

// Tile geometry: one CTA per SM computes 128 x 256 output tiles with K
// slices of 64 (one 128-byte swizzle row of bf16), 4-stage smem ring.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 256;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBN * kBK * 2;
constexpr uint32_t kTmemCols = 512;   // two 128 x 256 fp32 accumulators
constexpr int kSmemBytes = kStages * (kABytes + kBBytes) + 1024 /*barriers*/ + 1024 /*align slack*/;
// Epilogue warps of each CTA of the pair kernel.  In GEMM -> ReduceScatter
// they form two groups of half of them, one per accumulator, and each warp
// of a group signals its share of a finished tile on its own.
constexpr int kPairEpiWarps = 8;

// Status word sites (which wait gave up), reported by cm_check_status.
enum Site : uint32_t {
    kSiteProducerFlag = 1,
    kSiteForwardFlag = 2,
    kSiteEpilogueFlag = 3,
    kSiteEmpty = 4,
    kSiteFull = 5,
    kSiteTmemEmpty = 6,
    kSiteTmemFull = 7,
    kSiteForwardFull = 8,
    // debug builds (CM_DEBUG_BOUNDS): which computed index fell outside its buffer
    kSiteBoundsFlag = 16,
    kSiteBoundsForward = 17,
    kSiteBoundsOutput = 18,
    kSiteBoundsBucket = 19,
    kSiteBoundsSlab = 20,
    kSiteBoundsTask = 21,
};

struct KParams {
    CUtensorMap tmA0;   // x: AG shards / RS per-rank row slabs, as [slabs*chunks][rows_c][K]
    CUtensorMap tmA1;   // AG workspace receive slots, same view (loads and forward stores)
    CUtensorMap tmB;    // weights: [N][n][K] (K-major) or [N][K][n] (n-major)
    CUtensorMap tmAcc;  // RS fp32 accumulators as [bufs*chunks][rows_c][n], 32 x 32 boxes (CTA pairs)
    CUtensorMap tmAccIn;  // the same view, 32-column x pre_box_rows boxes: received buckets
                          // loaded through the operand ring (rs_preload)
    void *y;
    float *acc;                // RS circulating accumulators
    int bucket_hint;           // CTA pairs, TMA RS epilogue: L2 policy of bucket writes and adds
                               // (0 none, 1 evict_first, 2 evict_last; CM_OPT_RS_BUCKET_HINT)
    uint32_t *flags;
    uint32_t *status;
    uint32_t *tile_counter;    // dynamic tile scheduler (CTA-pair kernel), zero at launch
    int static_tiles;          // CTA-pair kernel: 1 = cluster c takes tiles c, c + clusters, ...
                               // instead of the next index of the global counter
    int l2_hint_a, l2_hint_b;  // CTA-pair kernel: L2 priority of A / B loads (0 normal, 1 evict_last, 2 evict_first)
    int row_band;              // row tiles per band of the tile order (0 = a whole task group)
    int col_slabs;             // > 1: the tile order makes this many passes over the tasks, each over
                               // one slab of ntiles / col_slabs column tiles (ntiles a multiple of it)
    int q_only;                // >= 0: this launch covers only chunk q_only of every task
    const uint8_t *x_bytes;    // AG: x and the receive slots as bytes (pair forwarder)
    uint8_t *slot_bytes;
    int64_t row_bytes;         // bytes per A row (K * 2)
    int64_t y_rank_stride;     // AG: elements between Y_r and Y_{r+1}
    int64_t out_rows_per_idx;  // AG: rows per shard id (m, or N*m undecomposed); RS: rows per bucket
    int64_t acc_buf_stride;    // RS: elements per accumulator buffer
    uint64_t timeout_ns;
    int op;                    // 0 AllGather->GEMM, 1 GEMM->ReduceScatter
    int N, chunks;
    int rows_c;                // rows per chunk
    int mtiles_c, ntiles, kblocks;
    int n;
    int y_f32;
    int a_box_rows;
    int rs_preload;            // RS, CTA pairs of one cluster: received buckets preloaded into TMEM
    int pre_stages;            // ... as this many ring stages per tile (4: every slice, 2: the first two
                               //     32-column slices of each epilogue warp)
    int pre_box_rows;          // rows of a tmAccIn box (128, or rows_c if smaller)
    int rs_epi;                // CTA pairs, RS epilogue: 0 = every epilogue warp on every tile, TMA
                               // copies; 1 = two epilogue warp groups (one per accumulator) with vector
                               // reductions; 2 = every epilogue warp on every tile, vector reductions
    int chunk_pair;            // CTA pairs: a pair tile covers chunks 2g and 2g+1 (one per CTA; chunks
                               // of at most 128 rows), and the tile decode's chunk index is g
    int tiles_per_task, task_begin, task_end;
    uint32_t tgt_in, tgt_free;
    // extents the bounds checks of debug builds compare computed indices with
    int64_t flag_words;        // readiness counters after p.flags
    int64_t x_total;           // bytes of x (AG, the forwarder's source for step 0)
    int64_t slot_total;        // bytes of the receive slots (AG)
    int64_t y_elems;           // elements of the output
    int acc_bufs;              // RS accumulator buffers of acc_buf_stride elements
    int a0_slabs, a1_slabs, b_slabs;   // third extent of tmA0, tmA1, tmB
    cm_task tasks[kMaxTasks];
};

// Single-CTA kernel (128 x 256 tiles): launch for tasks [p.task_begin, p.task_end).
cudaError_t launch_persistent(const KParams &p, bool b_mn_major, int grid, cudaStream_t stream);

// One-time per-device kernel attributes; returns the SM count.
cudaError_t prepare_device(int device, int *num_sms);

// CTA-pair kernel (256 x 256 tiles; one pair per cluster).
int pair_rows();
cudaError_t prepare_pair(int device, int *max_clusters);
// layout: bit 0 = B MN-major, bit 1 = A MN-major.
cudaError_t launch_pair(const KParams &p, int layout, int clusters, cudaStream_t stream);
// Pipelined GEMM -> ReduceScatter: y rows of chunk j of every bucket = the sum
// over ranks of the fp32 partials P [N*N][Mb][n] (cm_reduce.cu).
cudaError_t launch_reduce_chunk(const float *P, void *y, int N, int64_t Mb, int64_t rc, int64_t n, int j, bool y_f32,
                                int sms, cudaStream_t stream);

}  // namespace cm
