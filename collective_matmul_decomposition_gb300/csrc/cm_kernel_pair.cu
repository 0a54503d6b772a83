// cm_kernel_pair.cu -- the persistent kernel on CTA pairs (tcgen05 .cta_group::2).
//
// Same task table and the same per-tile work as the single-CTA kernel, but
// every output tile is 256 x 256 and belongs to a pair of CTAs on two SMs:
// CTA c of the pair stages rows 128c..128c+127 of the A tile and columns
// 128c..128c+127 of the B tile, and one tcgen05.mma.cta_group::2 issued by the
// pair leader multiplies the whole 256-row tile into both CTAs' tensor memory
// (each CTA holds its 128 rows x 256 fp32 columns).  Each CTA fetches half the
// operand bytes per MMA of the single-CTA tile, so a 6-stage ring of 32 KB
// stages fits in shared memory.
//
// A cluster is one pair.  Every operand load is an ordinary TMA tile load
// into the loading CTA's own shared memory; no load is multicast.
//
// Tiles are handed out dynamically: a scheduler thread of the cluster leader
// takes the next tile index from a global counter and publishes it to every
// CTA through a small shared-memory queue, so clusters that finish early take the next
// tile in order (the tiles running at any time stay close together, which
// keeps their operands in L2) and a tile's dependencies are always on tiles
// handed out earlier.
//
// Roles (384 threads per CTA):
//   warp 0    producer: TMA loads of this CTA's halves.  All loads complete
//             on the pair leader's ring barrier; the leader posts the byte
//             count.
//   warp 3    scheduler (cluster leader only): takes tile j + 1 from the
//             global counter once the producer has started tile j, and
//             publishes it to every CTA of the cluster.
//   warp 1    MMA issuer (leader only): pair MMAs; commits each stage and,
//             per tile, the accumulator to the barriers of both CTAs.
//   warp 2    AG forwarder (both CTAs): every tile copies a slice of its CTA's
//             128 shard rows (1/column-tiles of them) to the ring neighbour's
//             receive slot with 1-D TMA bulk copies through four 8 KB buffers,
//             then bumps the slot's ready flag -- the rotation copy in flight
//             while the partial GEMMs read the shard.
//   warps 4-11  epilogue (both CTAs): 8 warps, TMEM lane quarter = warp % 4.
//             AG writes shard rows of Y_r (column half = (warp - 4) / 4).  RS
//             adds the tile into its bucket where the bucket lies (or, with
//             per-step buffers, adds the received bucket and stores the sum
//             to the next buffer); the owner rounds the complete bucket into
//             y.  Three arrangements (p.rs_epi): every warp on every tile
//             with TMA copies through a 4 KB swizzled buffer per warp; two
//             groups of four warps, one per TMEM accumulator, with coalesced
//             vector accesses; every warp on every tile with vector accesses.
//
// RS preload (p.pre_stages > 0): for a tile that receives a bucket, the
// scheduler acquires the bucket's flag before publishing the tile, the
// producer loads the CTA's rows of that bucket through the ring ahead of the
// K slices, and the MMA thread copies them into the accumulator
// (tcgen05.cp) and accumulates the partial GEMM onto them; the epilogue then
// only stores the preloaded slices.
// All waits are bounded; see cm_kernel.cu for the failure protocol.
#include <cuda_bf16.h>

#include "cm_kernel_common.cuh"

namespace cm {
namespace {

using namespace dev;
using namespace kc;

constexpr int kPairRows = 256;          // output rows per pair tile
constexpr int kCtaRows = 128;           // rows staged per CTA
constexpr int kPStages = 6;
constexpr int kPThreads = 384;
constexpr int kPEpiWarps = kPairEpiWarps;
constexpr int kHalfA = kCtaRows * kBK * 2;   // 16 KB
constexpr int kHalfB = (kBN / 2) * kBK * 2;  // 16 KB
constexpr int kFwdPiece = 8192;              // forwarder copy granule
constexpr int kFwdBufs = 4;                  // forwarder buffers (the same 32 KB as the RS epilogue's)
constexpr int kQueue = 6;                    // tile-index queue depth
constexpr int CL = 2;                        // CTAs per cluster: one pair
// RS preload: ring stage ps carries the 32-column fp32 boxes at columns
// 32*ps and 128 + 32*ps of the tile (slice ps of both epilogue column
// halves); p.pre_stages of them (2 or 4) precede the K slices.
constexpr int kPSmemBytes = kPStages * (kHalfA + kHalfB) + kFwdBufs * kFwdPiece + 1024 + 1024;

// Position of this CTA in its cluster.
struct Cl {
    uint32_t rank;     // %cluster_ctarank (0 = pair leader, issues the MMAs; 1 = its peer)
    uint32_t pos;      // same as rank
    uint32_t leader;   // cluster rank of the pair leader (0)
};

struct PSmem {
    uint8_t *a0, *b0;   // ring stage 0 of A and B; stage i is kHalfA (kHalfB) bytes further
    uint8_t *fbuf[1];   // AG: kFwdBufs forwarder copy buffers of kFwdPiece bytes from fbuf[0]; RS: the
                        // same 32 KB as 8 epilogue-warp buffers
    uint64_t *full, *empty, *tfull, *tempty, *drain, *fbar, *qfull, *qempty, *ebar, *started;
    int32_t *qent;      // tile queue: kQueue entries of kQWords words, each CTA its own (see QTile)
    uint32_t *tmem_slot;
    volatile int *abort;
};

// Consumer side of the tile queue: returns the next tile index (-1 = no more
// work or failure) and releases the slot on the leader.
// One published tile as a CTA sees it, worked out once by the cluster
// leader's scheduler: the tile (-1 = no more work or failure), where it lies,
// and this CTA's load coordinates for its first K slice.
struct QTile {
    int t, task, q, mt, nt, nk, a_src, a_row, n0, slab, rr, sig;
    int pre;        // RS preload: accumulator buffer whose bucket is loaded before the K slices, -1 none
    int row0;       // this CTA's first output row inside its chunk q
    int ready;      // RS: the scheduler found every input flag of the tile already at its target
    int pad;
};
constexpr int kQWords = 16;

// Consumer side of the tile queue.  Slots are released by the epilogue
// warps and (AG) the forwarders only: an epilogue warp reads entry j after
// the MMAs of tile j completed, which needed the producers' loads and the
// MMA thread's reads of that entry, so its release covers theirs.
struct QueueReader {
    int slot = 0;
    uint32_t phase = 0;
    uint32_t qempty_leader0;   // slot i's release barrier on the leader: 8*i bytes further

    __device__ void init(const PSmem &s) { qempty_leader0 = mapa_shared(smem_u32(&s.qempty[0]), 0); }
    __device__ QTile next(const KParams &p, const PSmem &s, bool release) {
        QTile e;
        e.t = -1;
        if (mbar_try_wait_cluster(&s.qfull[slot], phase) ||
            wait_mbar<true>(p, s.abort, &s.qfull[slot], phase, kSiteEmpty, -1, -1)) {
            const volatile int4 *v = reinterpret_cast<const volatile int4 *>(s.qent + kQWords * slot);
            const int4 a = const_cast<const int4 &>(v[0]), b = const_cast<const int4 &>(v[1]),
                       c = const_cast<const int4 &>(v[2]), d = const_cast<const int4 &>(v[3]);
            e = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
        }
        if (release) mbar_arrive_cluster(qempty_leader0 + 8u * uint32_t(slot));
        if (++slot == kQueue) {
            slot = 0;
            phase ^= 1u;
        }
        return e;
    }
};

// Ring-barrier wait.  `ready` is a non-blocking test of the same barrier
// made right after the previous stage was handled, so its latency overlaps
// that stage's work; only when it said "not yet" is the barrier waited on.
__device__ __forceinline__ bool ring_wait(const KParams &p, volatile int *abort, uint64_t *bar, uint32_t parity,
                                          bool ready, uint32_t site, int task, int q) {
    if (ready || mbar_try_wait(bar, parity)) return true;
    return wait_mbar<false>(p, abort, bar, parity, site, task, q);
}

// LAYOUT bit 0: B is MN-major (W stored [K][n]); bit 1: A is MN-major (A
// stored [K][rows], rows contiguous -- a transposed activation, as in a
// weight-gradient GEMM).  An MN-major operand half is two 64-wide boxes.
template <int LAYOUT>
__device__ void producer(const KParams &p, const PSmem &s, int total, const Cl &cl) {
    constexpr bool B_MN = (LAYOUT & 1) != 0, A_MN = (LAYOUT & 2) != 0;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0;   // ring stages filled so far
    // the leader's ring barrier of stage i sits 8*i bytes after stage 0's
    const uint32_t full_leader0 = mapa_shared(smem_u32(&s.full[0]), cl.leader);
    const uint32_t a_smem0 = smem_u32(s.a0);
    const uint32_t b_smem0 = smem_u32(s.b0);
    // bytes per stage for the pair: each CTA's A half (one box) and B half
    const uint32_t a_half = uint32_t(p.a_box_rows) * kBK * 2;
    const uint32_t tx_pair = 2u * (a_half + kHalfB);
    auto policy = [](int h) {
        return h == 1 ? policy_evict_last() : h == 2 ? policy_evict_first() : policy_evict_normal();
    };
    const uint64_t pol_a = policy(p.l2_hint_a), pol_b = policy(p.l2_hint_b);
    const bool hinted = p.l2_hint_a != 0 || p.l2_hint_b != 0;
    const uint64_t tm_b = reinterpret_cast<uint64_t>(&p.tmB);
    QueueReader qr;
    qr.init(s);
    // tile indices come from the cluster leader's scheduler thread through
    // the queue; this CTA's producer tells it when a tile starts loading
    const bool signals = cl.rank == 0;
    const uint64_t tm_a0 = reinterpret_cast<uint64_t>(&p.tmA0), tm_a1 = reinterpret_cast<uint64_t>(&p.tmA1);
    const int slab_step = p.N * p.chunks;
    QTile c = qr.next(p, s, false);
    while (c.t >= 0 && !*s.abort) {
        // A rows that arrived by the ring were acquired by the scheduler
        // before it published this entry; order them before our TMA reads
        if (c.a_src == 1) fence_proxy_async_global();
        // Slice coordinates.  A: (K offset, row, slab); B: (K offset, column,
        // rank), or (column, K offset, rank) when W is MN-major.  A tile that
        // sums over ranks (a_src 2) walks rank by rank through the K slices.
        int rr = c.rr, slab = c.slab;
        const uint64_t tm_a = c.a_src == 1 ? tm_a1 : tm_a0;
        const int a_row = c.a_row, n0 = c.n0, nk = c.nk;
        if (kCheckBounds) {
            const int runs = (nk + p.kblocks - 1) / p.kblocks;   // ranks a summed tile walks through
            const int a_lim = c.a_src == 1 ? p.a1_slabs : p.a0_slabs;
            in_bounds(p, slab >= 0 && slab + (runs - 1) * slab_step < a_lim && rr >= 0 && rr + runs - 1 < p.b_slabs,
                      kSiteBoundsSlab, c.task, c.q);
        }
        int kb = 0;
        bool ok = true;
        bool free_ready = mbar_test_wait(s.empty + stage, phase ^ 1u);
        if (c.pre >= 0) {
            // RS preload: this CTA's 128 rows x 256 columns of the received
            // bucket, ahead of the K slices, through the same ring; the
            // scheduler acquired its flag before publishing this entry
            fence_proxy_async_global();
            const uint32_t tx_pre = 2u * 2u * uint32_t(p.pre_box_rows) * 128u;   // two boxes on each CTA
            const uint64_t tm_pre = reinterpret_cast<uint64_t>(&p.tmAccIn);
            const int pslab = c.pre * p.chunks + c.q;
            for (int ps = 0; ps < p.pre_stages; ++ps) {
                if (!ring_wait(p, s.abort, s.empty + stage, phase ^ 1u, free_ready, kSiteEmpty, c.task, c.q)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = full_leader0 + 8u * uint32_t(stage);
                const uint32_t sa = a_smem0 + uint32_t(stage) * kHalfA, sb = b_smem0 + uint32_t(stage) * kHalfB;
                const int col = c.nt * kBN + 32 * ps;
                if (cl.pos == 0) mbar_expect_tx(s.full + stage, tx_pre);
                tma_load_3d_pair_a(sa, tm_pre, fb, col, a_row, pslab);
                tma_load_3d_pair_a(sb, tm_pre, fb, col + kBN / 2, a_row, pslab);
                ++issued;
                if (++stage == kPStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                free_ready = mbar_test_wait(s.empty + stage, phase ^ 1u);
            }
        }
        for (int kk = 0; kk < nk && ok; ++kk) {
            if (!ring_wait(p, s.abort, s.empty + stage, phase ^ 1u, free_ready, kSiteEmpty, c.task, c.q)) {
                ok = false;
                break;
            }
            const uint32_t fb = full_leader0 + 8u * uint32_t(stage);
            const uint32_t sa = a_smem0 + uint32_t(stage) * kHalfA, sb = b_smem0 + uint32_t(stage) * kHalfB;
            const int k0 = kb * kBK;
            if (cl.pos == 0) mbar_expect_tx(s.full + stage, tx_pair);
            if (A_MN) {
                for (int j = 0; j < kCtaRows / 64; ++j)
                    tma_load_3d_pair_a(sa + uint32_t(j * (64 * kBK * 2)), tm_a, fb, a_row + 64 * j, k0, slab);
            } else if (hinted)
                tma_load_3d_pair_hint_a(sa, tm_a, fb, k0, a_row, slab, pol_a);
            else
                tma_load_3d_pair_a(sa, tm_a, fb, k0, a_row, slab);
            if (B_MN) {
                for (int j = 0; j < kBN / 2 / 64; ++j)
                    tma_load_3d_pair_a(sb + uint32_t(j * (64 * kBK * 2)), tm_b, fb, n0 + 64 * j, k0, rr);
            } else if (hinted) {
                tma_load_3d_pair_hint_a(sb, tm_b, fb, k0, n0, rr, pol_b);
            } else {
                tma_load_3d_pair_a(sb, tm_b, fb, k0, n0, rr);
            }
            ++issued;
            if (++stage == kPStages) {
                stage = 0;
                phase ^= 1u;
            }
            free_ready = mbar_test_wait(s.empty + stage, phase ^ 1u);
            if (++kb == p.kblocks) {
                kb = 0;
                ++rr;
                slab += slab_step;
            }
            if (signals && kk == 0) mbar_arrive(s.started);
        }
        if (!ok) break;
        c = qr.next(p, s, false);
    }
    // a pair leader's ring barriers count every load into its pair: once they
    // complete, no load is still writing this pair's shared memory.  Stage i
    // was last filled in the current round of the ring if i < stage, else in
    // the round before (if it was filled at all).
    if (cl.pos == 0)
        for (int i = 0; i < kPStages; ++i)
            if (uint32_t(i) < issued) drain_mbar<true>(p, &s.full[i], i < stage ? phase : phase ^ 1u);
}

// The cluster leader's scheduler (warp 3): takes tile indices from the
// global counter (or the next of its static round-robin share), decodes each
// once, works out every CTA's load coordinates, waits until an AG tile's A
// rows have arrived, and publishes a ready-to-use entry to every CTA of the
// cluster.  Tile j + 1 is taken once the leader's producer has started
// loading tile j, so a cluster holds at most one tile beyond the one loading,
// and none of this sits on the producer's path between two tiles.
__device__ void scheduler(const KParams &p, const PSmem &s, int total) {
    const int cid = int(blockIdx.x) / CL, ncl = int(gridDim.x) / CL;
    int static_next = cid, slot = 0;
    uint32_t qphase = 0, sphase = 0;
    for (int j = 0;; ++j) {
        if (j > 0) {
            if (!wait_mbar<false>(p, s.abort, s.started, sphase, kSiteEmpty, -1, -1)) return;
            sphase ^= 1u;
        }
        int t;
        if (p.static_tiles) {
            t = static_next;
            static_next += ncl;
        } else {
            t = int(atomic_add_relaxed(p.tile_counter, 1u));
        }
        if (t >= total) t = -1;
        TileCoord c = {0, 0, 0, 0};
        if (t >= 0) c = decode(p, t);
        if (t >= 0 && !in_bounds(p, c.task >= p.task_begin && c.task < p.task_end && c.q >= 0 && c.q < p.chunks,
                                 kSiteBoundsTask, c.task, c.q)) {
            t = -1;   // publish the end: nothing of this tile is loaded, computed or stored
            c = {p.task_begin, 0, 0, 0};
        }
        const cm_task &tk = p.tasks[c.task];
        // AG: the tile's A rows arrive by the ring; the producers that read
        // this entry see them (acquire here, release to them by the queue)
        // the chunks this tile reads: c.q, or 2*c.q and 2*c.q + 1 when a pair
        // tile covers two chunks (one per CTA)
        const int q0 = p.chunk_pair ? 2 * c.q : c.q, nq = p.chunk_pair ? 2 : 1;
        if (t >= 0 && p.op == 0 && tk.wait_in[0] >= 0)
            for (int qq = q0; qq < q0 + nq; ++qq)
                if (!wait_flag(p, s.abort, flag_ptr(p, tk.wait_in[0], qq, c.mt, c.nt), p.tgt_in, kSiteProducerFlag,
                               c.task, qq))
                    return;
        // RS preload: the received bucket is read before the partial GEMM, so
        // its producers must be done before this tile is published
        const bool pre = t >= 0 && p.op == 1 && p.rs_preload && p.pre_stages > 0 && tk.in_buf[0] >= 0 &&
                         tk.in_buf[0] != tk.out_buf;
        if (pre && tk.wait_in[0] >= 0)
            for (int qq = q0; qq < q0 + nq; ++qq)
                if (!wait_flag(p, s.abort, flag_ptr(p, tk.wait_in[0], qq, c.mt, c.nt), p.tgt_in, kSiteProducerFlag,
                               c.task, qq))
                    return;
        // RS: one look (no waiting) at the flags the tile's epilogue would wait
        // for; if all are complete the epilogue skips its wait
        int ready = 1;
        if (t >= 0 && p.op == 1) {
            for (int jj = 0; jj < 2 && ready; ++jj)
                if (tk.wait_in[jj] >= 0 && !(pre && jj == 0))
                    for (int qq = q0; qq < q0 + nq && ready; ++qq)
                        if (ld_acquire(flag_ptr(p, tk.wait_in[jj], qq, c.mt, c.nt)) < p.tgt_in) ready = 0;
            if (tk.wait_free[0] >= 0) ready = 0;
        }
        if (!wait_mbar<true>(p, s.abort, &s.qempty[slot], qphase ^ 1u, kSiteEmpty, -1, -1)) return;
        const bool sum_ranks = tk.a_src == 2;
        const int slab0 = (sum_ranks ? tk.out_idx : tk.a_slab) * p.chunks;
        const int rr = sum_ranks ? 0 : tk.rank;
        const int nk = kslices(p, tk), sig = p.op == 0 ? tk.sig_done : -1;
        for (uint32_t r = 0; r < uint32_t(CL); ++r) {
            const int pos = int(r);
            const int nt = c.nt;
            const int q = p.chunk_pair ? q0 + pos : c.q;   // this CTA's chunk
            const int row0 = p.chunk_pair ? 0 : c.mt * kPairRows + pos * kCtaRows;
            const int a_row = row0;
            const int slab = slab0 + q;
            const int n0 = nt * kBN + pos * (kBN / 2);
            int32_t *e = s.qent + kQWords * slot;
            const uint32_t w[kQWords] = {uint32_t(t),   uint32_t(c.task), uint32_t(q),   uint32_t(c.mt),
                                         uint32_t(nt),  uint32_t(nk),     uint32_t(tk.a_src), uint32_t(a_row),
                                         uint32_t(n0),  uint32_t(slab),   uint32_t(rr),       uint32_t(sig),
                                         uint32_t(pre ? int(tk.in_buf[0]) : -1), uint32_t(row0), uint32_t(ready), 0u};
            if (r == 0) {
                for (int i = 0; i < kQWords; ++i) e[i] = int32_t(w[i]);
            } else {
                const uint32_t ra = mapa_shared(smem_u32(e), r);
                for (int i = 0; i < kQWords; i += 4) st_shared_cluster_v4(ra + 4u * i, w[i], w[i + 1], w[i + 2], w[i + 3]);
            }
        }
        mbar_arrive(&s.qfull[slot]);
        for (uint32_t r = 1; r < uint32_t(CL); ++r) mbar_arrive_cluster(mapa_shared(smem_u32(&s.qfull[slot]), r));
        if (++slot == kQueue) {
            slot = 0;
            qphase ^= 1u;
        }
        if (t < 0) return;
    }
}

template <int LAYOUT>
__device__ void mma_issuer(const KParams &p, const PSmem &s, uint32_t tmem_base, const Cl &cl) {
    constexpr bool B_MN = (LAYOUT & 1) != 0, A_MN = (LAYOUT & 2) != 0;
    constexpr uint32_t kIdesc = idesc_bf16(kPairRows, kBN, B_MN, A_MN);
    // SW128 descriptors: K-major halves step 32 bytes per K=16 MMA; MN-major
    // halves are two 64-wide blocks 8 KB apart and step 16 rows of 128 bytes
    constexpr uint32_t kALbo = A_MN ? 64 * kBK * 2 : 16;
    constexpr uint32_t kAStep = A_MN ? (16 * 128) >> 4 : 32 >> 4;
    constexpr uint32_t kBLbo = B_MN ? 64 * kBK * 2 : 16;
    constexpr uint32_t kBStep = B_MN ? (16 * 128) >> 4 : 32 >> 4;
    // descriptors of ring stage 0; stage i adds its byte offset / 16 to the
    // start-address field (shared addresses stay below 2^18, so no carry)
    const uint64_t ad0 = desc_sw128(smem_u32(s.a0), kALbo, 1024);
    const uint64_t bd0 = desc_sw128(smem_u32(s.b0), kBLbo, 1024);
    // RS preload stages hold fp32 boxes of 128 rows x 128 bytes, SW128
    const uint64_t pd_a0 = desc_sw128(smem_u32(s.a0), 16, 1024);
    const uint64_t pd_b0 = desc_sw128(smem_u32(s.b0), 16, 1024);
    QueueReader qr;
    qr.init(s);
    int stage = 0;
    uint32_t phase = 0;
    int accb = 0;
    uint32_t acc_phase = 0;
    for (;;) {
        const QTile c = qr.next(p, s, false);
        if (c.t < 0 || *s.abort) break;
        if (!mbar_try_wait_cluster(&s.tempty[accb], acc_phase ^ 1u) &&
            !wait_mbar<true>(p, s.abort, &s.tempty[accb], acc_phase ^ 1u, kSiteTmemEmpty, c.task, c.q))
            break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(accb * kBN);
        const int nk = c.nk;
        bool ok = true;
        bool full_ready = mbar_test_wait(s.full + stage, phase);
        // RS preload: copy the received bucket into the accumulator; the
        // partial GEMM then adds onto it
        const int npre = c.pre >= 0 ? p.pre_stages : 0;
        for (int ps = 0; ps < npre; ++ps) {
            if (!ring_wait(p, s.abort, s.full + stage, phase, full_ready, kSiteFull, c.task, c.q)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t pa = pd_a0 + uint64_t((uint32_t(stage) * kHalfA) >> 4);
            const uint64_t pb = pd_b0 + uint64_t((uint32_t(stage) * kHalfB) >> 4);
            const uint32_t col = d + uint32_t(32 * ps);
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_cp_pair_128x256b(col + uint32_t(8 * j), pa + uint64_t(2 * j));
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_cp_pair_128x256b(col + uint32_t(kBN / 2 + 8 * j), pb + uint64_t(2 * j));
            mma_commit_pair_mc(s.empty + stage, uint16_t((1u << CL) - 1u));
            if (++stage == kPStages) {
                stage = 0;
                phase ^= 1u;
            }
            full_ready = mbar_test_wait(s.full + stage, phase);
        }
        const uint32_t acc0 = npre > 0 ? 1u : 0u;
        for (int kk = 0; kk < nk && ok; ++kk) {
            if (!ring_wait(p, s.abort, s.full + stage, phase, full_ready, kSiteFull, c.task, c.q)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t ad = ad0 + uint64_t((uint32_t(stage) * kHalfA) >> 4);
            const uint64_t bd = bd0 + uint64_t((uint32_t(stage) * kHalfB) >> 4);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
                mma_bf16_pair(d, ad + uint64_t(kAStep * k), bd + uint64_t(kBStep * k), kIdesc, (kk | k) != 0 ? 1u : acc0);
            mma_commit_pair_mc(s.empty + stage, uint16_t((1u << CL) - 1u));   // every CTA's stage s
            if (++stage == kPStages) {
                stage = 0;
                phase ^= 1u;
            }
            full_ready = mbar_test_wait(s.full + stage, phase);
        }
        if (!ok) break;
        mma_commit_pair_mc(&s.tfull[accb], uint16_t((1u << CL) - 1u));   // both CTAs' accumulators
        // AG: both CTAs' A slices of this tile have landed; the slot rows may be reused
        if (c.sig >= 0) {
            red_release_add(flag_ptr(p, c.sig, c.q, c.mt, c.nt), 1u);
            if (p.chunk_pair) red_release_add(flag_ptr(p, c.sig, c.q + 1, c.mt, c.nt), 1u);   // the peer CTA's chunk
        }
        if (++accb == 2) {
            accb = 0;
            acc_phase ^= 1u;
        }
    }
    mma_commit_pair(s.drain);
    drain_mbar<true>(p, s.drain, 0);
}

__device__ void forwarder(const KParams &p, const PSmem &s, const Cl &cl) {
    QueueReader qr;
    qr.init(s);
    uint32_t fph = 0;   // bit b: the phase of buffer b's barrier
    // every tile of a row tile forwards a slice of the rows: column tile nt
    // copies rows [nt*per, (nt+1)*per) of this CTA's 128, so the shard chunk
    // moves while all its tiles run instead of one tile doing all of it
    const int per = (kCtaRows + p.ntiles - 1) / p.ntiles;
    for (;;) {
        const QTile c = qr.next(p, s, true);
        if (c.t < 0 || *s.abort) break;
        const cm_task &tk = p.tasks[c.task];
        if (!(tk.fwd_slot[0] >= 0 || tk.fwd_slot[1] >= 0)) continue;
        bool ok = true;
        if (tk.a_src == 1 && tk.wait_in[0] >= 0)   // the shard chunk has arrived here
            ok = wait_flag(p, s.abort, flag_ptr(p, tk.wait_in[0], c.q, c.mt, c.nt), p.tgt_in, kSiteForwardFlag,
                           c.task, c.q);
        if (!ok) break;
        fence_proxy_async_global();
        const int lo = c.nt * per;
        const int row0 = c.row0 + lo;
        const int nrows = min(min(per, kCtaRows - lo), p.rows_c - row0);
        if (nrows > 0) {
            const int64_t rb = p.row_bytes;
            const uint8_t *src = (tk.a_src == 1 ? p.slot_bytes : p.x_bytes) +
                                 (int64_t(tk.a_slab * p.chunks + c.q) * p.rows_c + row0) * rb;
            uint8_t *dst[2] = {nullptr, nullptr};
            for (int j = 0; j < 2; ++j)
                if (tk.fwd_slot[j] >= 0)
                    dst[j] = p.slot_bytes + (int64_t(tk.fwd_slot[j] * p.chunks + c.q) * p.rows_c + row0) * rb;
            const int64_t bytes = int64_t(nrows) * rb;
            if (kCheckBounds) {
                const uint8_t *sb = tk.a_src == 1 ? p.slot_bytes : p.x_bytes;
                const int64_t st = tk.a_src == 1 ? p.slot_total : p.x_total;
                bool okb = src >= sb && src - sb + bytes <= st;
                for (int j = 0; j < 2; ++j)
                    if (dst[j]) okb = okb && dst[j] >= p.slot_bytes && dst[j] - p.slot_bytes + bytes <= p.slot_total;
                if (!in_bounds(p, okb, kSiteBoundsForward, c.task, c.q)) break;
            }
            // pieces go through kFwdBufs buffers: up to kFwdBufs loads in
            // flight, each buffer refilled once the store of its previous
            // piece has read it
            const int np = int((bytes + kFwdPiece - 1) / kFwdPiece);
            auto piece = [&](int i) { return uint32_t(min(int64_t(kFwdPiece), bytes - int64_t(i) * kFwdPiece)); };
            auto fbuf = [&](int b) { return s.fbuf[0] + b * kFwdPiece; };
            auto load = [&](int i) {
                const int b = i % kFwdBufs;
                mbar_expect_tx(&s.fbar[b], piece(i));
                bulk_load(fbuf(b), src + int64_t(i) * kFwdPiece, piece(i), &s.fbar[b]);
            };
            int issued = min(np, kFwdBufs);
            for (int i = 0; i < issued; ++i) load(i);
            for (int i = 0; i < np && ok; ++i) {
                const int b = i % kFwdBufs;
                ok = wait_mbar<false>(p, s.abort, &s.fbar[b], (fph >> b) & 1u, kSiteForwardFull, c.task, c.q);
                if (!ok) {
                    // leaving early: pieces i .. issued - 1 (one per buffer)
                    // may still be landing in this CTA's buffers
                    for (int j = i; j < issued; ++j) {
                        const int bj = j % kFwdBufs;
                        drain_mbar<false>(p, &s.fbar[bj], (fph >> bj) & 1u);
                    }
                    break;
                }
                fph ^= 1u << b;
                for (int j = 0; j < 2; ++j)
                    if (dst[j]) bulk_store(dst[j] + int64_t(i) * kFwdPiece, fbuf(b), piece(i));
                bulk_commit();
                if (i >= 1 && issued < np) {
                    bulk_wait_read<1>();   // every store but piece i's has read its buffer: piece i-1's is free
                    load(issued++);
                }
            }
            bulk_wait<0>();   // the copies are complete in global memory
            if (!ok) break;
        }
        fence_proxy_async_global();
        for (int j = 0; j < 2; ++j)
            if (tk.fwd_slot[j] >= 0 && tk.sig_fwd[j] >= 0)
                red_release_add(flag_ptr(p, tk.sig_fwd[j], c.q, c.mt, c.nt), 1u);
    }
    bulk_wait<0>();
}

// One 32-column slice of one row of an AG tile: the shard's rows of Y_r
// (DynamicUpdateSlice), bf16 (RNE) or fp32.
__device__ __forceinline__ void ag_store_slice(const KParams &p, const cm_task &tk, int64_t crow, int col0,
                                               const uint32_t (&v)[32]) {
    const int64_t orow = int64_t(tk.rank) * p.y_rank_stride + (int64_t(tk.out_idx) * p.out_rows_per_idx + crow) * p.n;
    if (!in_bounds(p, orow >= 0 && orow + col0 + min(32, p.n - col0) <= p.y_elems, kSiteBoundsOutput, tk.rank,
                   tk.out_idx))
        return;
    if (p.y_f32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.y) + orow + col0);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (col0 + 4 * i < p.n)
                dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                     __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
    } else {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.y) + orow + col0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (col0 + 8 * i >= p.n) break;
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[8 * i + 2 * h]),
                                                          __uint_as_float(v[8 * i + 2 * h + 1]));
                w[h] = *reinterpret_cast<uint32_t *>(&b2);
            }
            dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// AllGather -> GEMM epilogue: each warp reads its 32 TMEM lanes x 128
// columns in 32-column slices and stores them into the shard's rows of Y_r.
__device__ void epilogue_ag(const KParams &p, const PSmem &s, uint32_t tmem_base, const Cl &cl) {
    const int e = int(threadIdx.x) / 32 - 4;   // 0..7
    const int lane = int(threadIdx.x) & 31;
    const int quad = e & 3;                      // TMEM lanes 32*quad.. (warp % 4)
    const int half = e >> 2;                     // columns 128*half..
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&s.tempty[0]), cl.leader);   // buffer b: +8*b
    QueueReader qr;
    if (lane == 0) qr.init(s);
    int accb = 0;
    uint32_t acc_phase = 0;
    for (;;) {
        QTile e;
        if (lane == 0) e = qr.next(p, s, true);
        const int t = __shfl_sync(0xffffffffu, e.t, 0);
        bool bad = t < 0;
        TileCoord c;
        c.task = bad ? 0 : __shfl_sync(0xffffffffu, e.task, 0);
        c.q = __shfl_sync(0xffffffffu, e.q, 0);
        c.mt = __shfl_sync(0xffffffffu, e.mt, 0);
        c.nt = __shfl_sync(0xffffffffu, e.nt, 0);
        const int row0 = __shfl_sync(0xffffffffu, e.row0, 0);   // this CTA's first row in chunk c.q
        const cm_task &tk = p.tasks[c.task];
        if (!bad) bad = !wait_mbar<true>(p, s.abort, &s.tfull[accb], acc_phase, kSiteTmemFull, c.task, c.q);
        bad = bar_or(1, kPEpiWarps * 32, bad || *s.abort != 0);
        if (bad) break;
        tc_fence_after();

        const int row = row0 + quad * 32 + lane;   // row inside the chunk
        const bool row_ok = row < p.rows_c;
        const int64_t crow = int64_t(c.q) * p.rows_c + row;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
            const int col_local = half * 128 + cb * 32;
            const int col0 = c.nt * kBN + col_local;
            uint32_t v[32];
            tmem_ld32(tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(accb * kBN + col_local), v);
            tmem_wait_ld();
            if (row_ok && col0 < p.n) ag_store_slice(p, tk, crow, col0, v);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader0 + 8u * uint32_t(accb));
        if (++accb == 2) {
            accb = 0;
            acc_phase ^= 1u;
        }
    }
}


// L2 policy of bucket writes and adds (CM_OPT_RS_BUCKET_HINT; unused at 0).
__device__ __forceinline__ uint64_t bucket_policy(const KParams &p) {
    return p.bucket_hint == 2 ? policy_evict_last() : policy_evict_first();
}

// Row `row` of a 32 x 32 fp32 box staged by TMA with the 128-byte swizzle:
// 16-byte chunk j of row r sits at chunk position j ^ (r & 7).
__device__ __forceinline__ float4 *swz_row(uint8_t *buf, int row) { return reinterpret_cast<float4 *>(buf + row * 128); }

// GEMM -> ReduceScatter epilogue through the TMA unit (CM_OPT_RS_EPILOGUE =
// 1).  All eight warps drain every tile: warp e takes 32 rows (TMEM lanes
// 32*(e % 4)..) x 128 columns (half e / 4), per 32-column slice (one 4 KB
// fp32 box staged in shared memory):
//  - a bucket kept in place (in_buf[0] == out_buf): the TMEM slice is added
//    into the bucket where it lies with a TMA reduce-add, so nothing comes
//    back to the SM;
//  - the first contributor (no input): the slice is TMA-stored as the bucket;
//  - a bucket in per-step buffers: the received partial bucket is TMA-loaded,
//    the slice added, and the sum TMA-stored to the next rank's buffer;
//  - the owner: the received partial bucket(s) are TMA-loaded, the slice
//    added, and the sum rounded into the output.
template <bool HINT>
__device__ void epilogue_rs_tma(const KParams &p, const PSmem &s, uint32_t tmem_base, const Cl &cl) {
    const int e = int(threadIdx.x) / 32 - 4;   // 0..7
    const int lane = int(threadIdx.x) & 31;
    const int quad = e & 3;
    const int half = e >> 2;
    const bool leader_thread = e == 0 && lane == 0;
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&s.tempty[0]), cl.leader);   // buffer b: +8*b
    uint8_t *buf = s.fbuf[0] + e * 4096;
    uint64_t *eb = &s.ebar[e];
    uint32_t eph = 0;
    bool store_pending = false;   // lane 0: a TMA store / reduce may still be reading buf
    QueueReader qr;
    if (lane == 0) qr.init(s);
    int accb = 0;
    uint32_t acc_phase = 0;
    for (;;) {
        QTile e;
        if (lane == 0) e = qr.next(p, s, true);
        const int t = __shfl_sync(0xffffffffu, e.t, 0);
        bool bad = t < 0;
        TileCoord c;
        c.task = bad ? 0 : __shfl_sync(0xffffffffu, e.task, 0);
        c.q = __shfl_sync(0xffffffffu, e.q, 0);
        c.mt = __shfl_sync(0xffffffffu, e.mt, 0);
        c.nt = __shfl_sync(0xffffffffu, e.nt, 0);
        const int row0 = __shfl_sync(0xffffffffu, e.row0, 0);   // this CTA's first row in chunk c.q
        const int pre = __shfl_sync(0xffffffffu, e.pre, 0);   // in_buf[0]'s slices cb < p.pre_stages are
                                                              // already in the accumulator
        const int ready = __shfl_sync(0xffffffffu, e.ready, 0);   // inputs found complete by the scheduler
        const cm_task &tk = p.tasks[c.task];
        if (!bad) bad = !wait_mbar<true>(p, s.abort, &s.tfull[accb], acc_phase, kSiteTmemFull, c.task, c.q);
        if (leader_thread && !bad && !ready) {
            for (int j = 0; j < 2 && !bad; ++j)
                if (tk.wait_in[j] >= 0)
                    bad = !wait_flag(p, s.abort, flag_ptr(p, tk.wait_in[j], c.q, c.mt, c.nt), p.tgt_in,
                                     kSiteEpilogueFlag, c.task, c.q);
            if (!bad && tk.wait_free[0] >= 0)
                bad = !wait_flag(p, s.abort, flag_ptr(p, tk.wait_free[0], c.q, c.mt, c.nt), p.tgt_free,
                                 kSiteEpilogueFlag, c.task, c.q);
        }
        bad = bar_or(1, kPEpiWarps * 32, bad || *s.abort != 0);
        if (bad) break;
        if (lane == 0) fence_proxy_async_global();   // the received buckets were released by other CTAs
        tc_fence_after();

        const int row_w = row0 + quad * 32;   // warp's first row in the chunk
        const int row = row_w + lane;
        const bool row_ok = row < p.rows_c;
        const int64_t crow = int64_t(c.q) * p.rows_c + row;
        // the bucket is accumulated where it lies: its partial sum is not read here
        const bool in_place = tk.out_buf >= 0 && tk.in_buf[0] == tk.out_buf;
        bool skip = false;   // a bucket load failed (the kernel is aborting): no further copies this tile
        if (kCheckBounds) {
            bool okb = tk.out_buf < p.acc_bufs && tk.in_buf[0] < p.acc_bufs && tk.in_buf[1] < p.acc_bufs;
            if (tk.out_buf < 0)
                okb = okb && (int64_t(tk.out_idx) * p.out_rows_per_idx + int64_t(c.q + 1) * p.rows_c) * p.n <= p.y_elems;
            skip = !in_bounds(p, okb, kSiteBoundsBucket, c.task, c.q);
        }
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
            const int col_local = half * 128 + cb * 32;
            const int col0 = c.nt * kBN + col_local;
            uint32_t v[32];
            tmem_ld32(tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(accb * kBN + col_local), v);
            tmem_wait_ld();
            if (skip || col0 >= p.n) continue;   // aborting, or the whole slice lies past the last column
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
            for (int j = 0; j < 2 && !skip; ++j) {
                if (tk.in_buf[j] < 0 || (j == 0 && (in_place || (pre >= 0 && cb < p.pre_stages)))) continue;
                if (lane == 0) {
                    if (store_pending) {
                        bulk_wait_read<0>();
                        store_pending = false;
                    }
                    mbar_expect_tx(eb, 32 * 32 * 4);
                    tma_load_3d(buf, &p.tmAcc, eb, col0, row_w, tk.in_buf[j] * p.chunks + c.q);
                }
                const bool landed = wait_mbar<false>(p, s.abort, eb, eph, kSiteEpilogueFlag, c.task, c.q);
                if (__any_sync(0xffffffffu, !landed)) {
                    // the load may still be landing in buf: wait for it (bounded) and stop
                    if (lane == 0) drain_mbar<false>(p, eb, eph);
                    skip = true;
                }
                eph ^= 1u;
                if (skip) break;
                float4 *r = swz_row(buf, lane);
#pragma unroll
                for (int i = 0; i < 8; ++i) add4(f + 4 * i, r[i ^ (lane & 7)]);
                __syncwarp();
            }
            if (skip) continue;
            if (tk.out_buf >= 0) {
                if (lane == 0 && store_pending) {
                    bulk_wait_read<0>();
                    store_pending = false;
                }
                __syncwarp();
                float4 *r = swz_row(buf, lane);
#pragma unroll
                for (int i = 0; i < 8; ++i) r[i ^ (lane & 7)] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int slab = tk.out_buf * p.chunks + c.q;
                    if (HINT) {
                        const uint64_t pol = bucket_policy(p);
                        if (in_place)
                            tma_reduce_add_3d_hint(&p.tmAcc, buf, col0, row_w, slab, pol);
                        else
                            tma_store_3d_hint(&p.tmAcc, buf, col0, row_w, slab, pol);
                    } else if (in_place) {
                        tma_reduce_add_3d(&p.tmAcc, buf, col0, row_w, slab);
                    } else {
                        tma_store_3d(&p.tmAcc, buf, col0, row_w, slab);
                    }
                    bulk_commit();
                    store_pending = true;
                }
            } else if (row_ok) {   // owner: the bucket is home
                const int64_t orow = (int64_t(tk.out_idx) * p.out_rows_per_idx + crow) * p.n;
                if (p.y_f32) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.y) + orow + col0);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (col0 + 4 * i < p.n) dst[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.y) + orow + col0);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (col0 + 8 * i >= p.n) break;
                        uint32_t w[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(f[8 * i + 2 * h], f[8 * i + 2 * h + 1]);
                            w[h] = *reinterpret_cast<uint32_t *>(&b2);
                        }
                        dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
        // half preload: the next tile in this buffer accumulates onto every
        // column, so the columns it will not preload must read zero
        if (p.pre_stages > 0 && p.pre_stages < 4) {
            for (int cb = p.pre_stages; cb < 4; ++cb)
                tmem_zero32(tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(accb * kBN + half * 128 + cb * 32));
            tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader0 + 8u * uint32_t(accb));
        if (tk.sig_done >= 0) {
            if (lane == 0) {
                bulk_wait<0>();            // this warp's bucket slices (stores or adds) are done in global memory
                store_pending = false;
                fence_proxy_async_global();
            }
            // every warp's copies are complete before the barrier; the
            // leader's release after it covers them (release is cumulative
            // over what the barrier orders before it), so no per-thread fence
            // is needed here (one measured 2 % slower on tiles of 4-24 K slices)
            bar_sync(1, kPEpiWarps * 32);
            if (leader_thread && !*s.abort) red_release_add(flag_ptr(p, tk.sig_done, c.q, c.mt, c.nt), 1u);
        }
        if (++accb == 2) {
            accb = 0;
            acc_phase ^= 1u;
        }
    }
    if (lane == 0) bulk_wait<0>();
}

// GEMM -> ReduceScatter epilogue with vector accesses, in one of two warp
// arrangements:
//  - GROUPS (CM_OPT_RS_EPILOGUE = 2): the eight epilogue warps form two
//    groups of four, one per TMEM accumulator: group g takes every other
//    tile (the ones the MMA thread put in accumulator g), so two tiles'
//    epilogues -- and their latencies (input flags, the wait for a tile's
//    adds to be performed) -- overlap.  Warp w reads TMEM lanes 32*(w % 4)..
//    and handles those 32 rows x 256 columns of the tile in eight 32-column
//    slices;
//  - all warps (CM_OPT_RS_EPILOGUE = 3): every warp on every tile, as the
//    TMA epilogue: warp w takes rows 32*(w % 4).. and columns 128*(w / 4)..
//    in four slices, so a tile drains in half the time of a group's.
// A slice read from TMEM (one row per lane) is turned round through the
// warp's 4 KB buffer, so that each lane then holds four consecutive columns
// of 8 rows and 8 lanes cover a row's 128 bytes: every global access below is
// a coalesced 16-byte vector, and none goes through the TMA unit, which stays
// free for the operand loads.
//  - a bucket kept in place (in_buf[0] == out_buf): the slice is added into
//    the bucket where it lies (red.global.add.v4.f32, performed at L2);
//  - the first contributor (no input): the slice is stored as the bucket;
//  - a bucket in per-step buffers: the received partial bucket is loaded,
//    the slice added, and the sum stored to the next rank's buffer;
//  - the owner: the received partial bucket(s) are loaded, the slice added,
//    and the sum rounded into the output.
// TMEM slices are loaded one ahead.  Each warp signals its share of a tile
// on its own, once its lanes' accesses are ordered before the signal (a
// fence in every lane, a warp barrier, a release by lane 0): a consumer waits
// for every warp that drains the tile (four or eight) in each CTA, and no
// warp waits for another.

template <bool GROUPS>
__device__ void epilogue_rs_vec(const KParams &p, const PSmem &s, uint32_t tmem_base, const Cl &cl) {
    constexpr int kSlices = GROUPS ? kBN / 32 : kBN / 64;   // 32-column slices per warp and tile
    const int e = int(threadIdx.x) / 32 - 4;   // 0..7
    const int lane = int(threadIdx.x) & 31;
    const int quad = e & 3;                    // TMEM lanes 32*quad.. (warp % 4)
    const int grp = e >> 2;                    // GROUPS: accumulator (and tile parity) of this warp's group;
                                               // else the warp's half of the tile's columns
    const int col_w = GROUPS ? 0 : grp * (kBN / 2);   // warp's first column in the tile
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&s.tempty[0]), cl.leader);   // buffer b: +8*b
    uint8_t *buf = s.fbuf[0] + e * 4096;   // 32 rows x 128 bytes; 16-byte chunk j of row r at j ^ (r & 7)
    const int tr = lane >> 3, tc = lane & 7;   // turned round: rows 4i + tr, columns 4tc..4tc+3 of the slice
    QueueReader qr;
    if (lane == 0) qr.init(s);
    int accb = GROUPS ? grp : 0;
    uint32_t acc_phase = 0;
    for (int j = 0;; ++j) {
        QTile e;
        if (lane == 0) e = qr.next(p, s, true);   // every warp reads (and releases) every entry
        const int t = __shfl_sync(0xffffffffu, e.t, 0);
        if (t < 0) break;
        if (GROUPS && (j & 1) != grp) continue;   // the other group's tile
        TileCoord c;
        c.task = __shfl_sync(0xffffffffu, e.task, 0);
        c.q = __shfl_sync(0xffffffffu, e.q, 0);
        c.mt = __shfl_sync(0xffffffffu, e.mt, 0);
        c.nt = __shfl_sync(0xffffffffu, e.nt, 0);
        const int row0 = __shfl_sync(0xffffffffu, e.row0, 0);   // this CTA's first row in chunk c.q
        const int pre = __shfl_sync(0xffffffffu, e.pre, 0);   // in_buf[0]'s slices with (slice % 4) <
                                                              // p.pre_stages are already in the accumulator
        const int ready = __shfl_sync(0xffffffffu, e.ready, 0);   // inputs found complete by the scheduler
        const cm_task &tk = p.tasks[c.task];
        bool bad = !wait_mbar<true>(p, s.abort, &s.tfull[accb], acc_phase, kSiteTmemFull, c.task, c.q);
        // each warp acquires the tile's input flags itself (unless the
        // scheduler already found them complete): no barrier across warps
        if (lane == 0 && !bad && !ready) {
            for (int jj = 0; jj < 2 && !bad; ++jj)
                if (tk.wait_in[jj] >= 0)
                    bad = !wait_flag(p, s.abort, flag_ptr(p, tk.wait_in[jj], c.q, c.mt, c.nt), p.tgt_in,
                                     kSiteEpilogueFlag, c.task, c.q);
            if (!bad && tk.wait_free[0] >= 0)
                bad = !wait_flag(p, s.abort, flag_ptr(p, tk.wait_free[0], c.q, c.mt, c.nt), p.tgt_free,
                                 kSiteEpilogueFlag, c.task, c.q);
        }
        bad = __any_sync(0xffffffffu, bad || *s.abort != 0);
        __syncwarp();   // lane 0's acquire orders the whole warp's accesses below
        if (bad) break;
        tc_fence_after();

        const int row_w = row0 + quad * 32;   // warp's first row in the chunk
        // the bucket is accumulated where it lies: its partial sum is not read here
        const bool in_place = tk.out_buf >= 0 && tk.in_buf[0] == tk.out_buf;
        const int64_t brow0 = int64_t(c.q) * p.rows_c + row_w;   // warp's first row in the bucket
        bool skip = false;   // debug builds: a buffer index outside its buffer; no global access this tile
        if (kCheckBounds) {
            bool okb = tk.out_buf < p.acc_bufs && tk.in_buf[0] < p.acc_bufs && tk.in_buf[1] < p.acc_bufs;
            if (tk.out_buf < 0)
                okb = okb && (int64_t(tk.out_idx) * p.out_rows_per_idx + int64_t(c.q + 1) * p.rows_c) * p.n <= p.y_elems;
            skip = !in_bounds(p, okb, kSiteBoundsBucket, c.task, c.q);
        }
        const uint32_t tcol = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(accb * kBN + col_w);
        uint32_t v[2][32];
        tmem_ld32(tcol, v[0]);
        tmem_wait_ld_regs(v[0]);
#pragma unroll
        for (int cb = 0; cb < kSlices; ++cb) {
            uint32_t(&cur)[32] = v[cb & 1];
            if (cb + 1 < kSlices) tmem_ld32(tcol + uint32_t((cb + 1) * 32), v[(cb + 1) & 1]);   // in flight
            const int col0 = c.nt * kBN + col_w + cb * 32;
            if (col0 < p.n && !skip) {
                float4 *wr = reinterpret_cast<float4 *>(buf + lane * 128);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    wr[k ^ (lane & 7)] = make_float4(__uint_as_float(cur[4 * k]), __uint_as_float(cur[4 * k + 1]),
                                                     __uint_as_float(cur[4 * k + 2]), __uint_as_float(cur[4 * k + 3]));
                __syncwarp();
                float4 x[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = 4 * i + tr;
                    x[i] = reinterpret_cast<const float4 *>(buf + r * 128)[tc ^ (r & 7)];
                }
                __syncwarp();   // every lane has read the buffer before the next slice is written
                const int col = col0 + 4 * tc;
                const bool col_ok = col < p.n;   // n is a multiple of 8: a vector is all in or all out
                for (int jj = 0; jj < 2; ++jj) {
                    if (tk.in_buf[jj] < 0 || (jj == 0 && (in_place || (pre >= 0 && (cb & 3) < p.pre_stages))))
                        continue;
                    const float *src = p.acc + int64_t(tk.in_buf[jj]) * p.acc_buf_stride + brow0 * p.n + col;
                    float4 a[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (col_ok && row_w + 4 * i + tr < p.rows_c)
                            a[i] = __ldcg(reinterpret_cast<const float4 *>(src + int64_t(4 * i + tr) * p.n));
                        else
                            a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        x[i].x += a[i].x;
                        x[i].y += a[i].y;
                        x[i].z += a[i].z;
                        x[i].w += a[i].w;
                    }
                }
                if (tk.out_buf >= 0) {
                    float *dst = p.acc + int64_t(tk.out_buf) * p.acc_buf_stride + brow0 * p.n + col;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (!col_ok || row_w + 4 * i + tr >= p.rows_c) continue;
                        float *d = dst + int64_t(4 * i + tr) * p.n;
                        if (in_place)
                            red_add_v4(d, x[i]);
                        else
                            __stcg(reinterpret_cast<float4 *>(d), x[i]);
                    }
                } else {   // owner: the bucket is home
                    const int64_t orow0 = (int64_t(tk.out_idx) * p.out_rows_per_idx + brow0) * p.n + col;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (!col_ok || row_w + 4 * i + tr >= p.rows_c) continue;
                        const int64_t o = orow0 + int64_t(4 * i + tr) * p.n;
                        if (p.y_f32) {
                            *reinterpret_cast<float4 *>(static_cast<float *>(p.y) + o) = x[i];
                        } else {
                            __nv_bfloat162 lo = __floats2bfloat162_rn(x[i].x, x[i].y);
                            __nv_bfloat162 hi = __floats2bfloat162_rn(x[i].z, x[i].w);
                            *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.y) + o) =
                                make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
                        }
                    }
                }
            }
            if (cb + 1 < kSlices) tmem_wait_ld_regs(v[(cb + 1) & 1]);
        }
        // half preload: the next tile in this accumulator adds onto every
        // column, so the columns it will not preload must read zero
        if (p.pre_stages > 0 && p.pre_stages < 4) {
            for (int h = GROUPS ? 0 : grp; h < (GROUPS ? 2 : grp + 1); ++h)
                for (int cb = p.pre_stages; cb < 4; ++cb)
                    tmem_zero32(tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(accb * kBN + h * 128 + cb * 32));
            tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty_leader0 + 8u * uint32_t(accb));
        if (tk.sig_done >= 0) {
            fence_acq_rel_gpu();   // this lane's adds / stores of the tile come before the signal
            __syncwarp();
            if (lane == 0 && !*s.abort) red_release_add(flag_ptr(p, tk.sig_done, c.q, c.mt, c.nt), 1u);
        }
        if (GROUPS) {
            acc_phase ^= 1u;
        } else if (++accb == 2) {
            accb = 0;
            acc_phase ^= 1u;
        }
    }
}

template <int LAYOUT>
__global__ void __launch_bounds__(kPThreads, 1) cm_pair_kernel(const __grid_constant__ KParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PSmem s;
    s.a0 = base;
    s.b0 = base + kPStages * kHalfA;
    s.fbuf[0] = base + kPStages * (kHalfA + kHalfB);
    uint64_t *bars = reinterpret_cast<uint64_t *>(s.fbuf[0] + kFwdBufs * kFwdPiece);
    s.full = bars;
    s.empty = s.full + kPStages;
    s.tfull = s.empty + kPStages;
    s.tempty = s.tfull + 2;
    s.drain = s.tempty + 2;
    s.fbar = s.drain + 1;
    s.qfull = s.fbar + kFwdBufs;
    s.qempty = s.qfull + kQueue;
    s.ebar = s.qempty + kQueue;
    s.started = s.ebar + kPEpiWarps;
    s.qent = reinterpret_cast<int32_t *>(s.started + 1);   // 16-byte aligned: 42 barriers precede it
    s.tmem_slot = reinterpret_cast<uint32_t *>(s.qent + kQWords * kQueue);
    s.abort = reinterpret_cast<volatile int *>(s.tmem_slot + 1);

    const int warp = int(threadIdx.x) >> 5, lane = int(threadIdx.x) & 31;
    Cl cl;
    cl.rank = cluster_ctarank();
    cl.pos = cl.rank;
    cl.leader = 0;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);   // the pair MMA's commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tfull[i], 1);
            // epilogue warps of both CTAs that drain accumulator i: all eight,
            // or the four of the group that owns it (RS in two groups)
            mbar_init(&s.tempty[i], 2 * (p.op == 1 && p.rs_epi == 1 ? kPEpiWarps / 2 : kPEpiWarps));
        }
        for (int i = 0; i < kFwdBufs; ++i) mbar_init(&s.fbar[i], 1);
        mbar_init(s.drain, 1);
        mbar_init(s.started, 1);
        // queue slot releases: 8 epilogue warps per CTA and (AG) both forwarders
        const uint32_t readers = CL * kPEpiWarps + (p.op == 0 ? CL : 0);
        for (int i = 0; i < kQueue; ++i) {
            mbar_init(&s.qfull[i], 1);
            mbar_init(&s.qempty[i], readers);
        }
        for (int i = 0; i < kPEpiWarps; ++i) mbar_init(&s.ebar[i], 1);
        *s.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&p.tmA0);
        prefetch_tmap(&p.tmA1);
        prefetch_tmap(&p.tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(s.tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers exist before any cross-CTA arrive or load
    tc_fence_after();
    const uint32_t tmem_base = *s.tmem_slot;
    const int total = (p.task_end - p.task_begin) * p.tiles_per_task;
    if (p.op == 1 && p.pre_stages > 0 && p.pre_stages < 4) {
        // half preload: both accumulators start with zeros in the columns
        // that are not preloaded (see the RS epilogue), before any MMA
        if (warp >= 4) {
            const int e = warp - 4;
            for (int b = 0; b < 2; ++b)
                for (int cb = p.pre_stages; cb < 4; ++cb)
                    tmem_zero32(tmem_base + (uint32_t((e & 3) * 32) << 16) +
                                uint32_t(b * kBN + (e >> 2) * 128 + cb * 32));
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();
        cluster_sync();
        tc_fence_after();
    }

    if (warp == 0) {
        if (lane == 0) producer<LAYOUT>(p, s, total, cl);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && cl.pos == 0) mma_issuer<LAYOUT>(p, s, tmem_base, cl);
        __syncwarp();
    } else if (warp == 2) {
        if (lane == 0 && p.op == 0) forwarder(p, s, cl);
        __syncwarp();
    } else if (warp == 3) {
        if (lane == 0 && cl.rank == 0) scheduler(p, s, total);
        __syncwarp();
    } else if (warp >= 4) {
        if (p.op == 0)
            epilogue_ag(p, s, tmem_base, cl);
        else if (p.rs_epi == 1)
            epilogue_rs_vec<true>(p, s, tmem_base, cl);
        else if (p.rs_epi == 2)
            epilogue_rs_vec<false>(p, s, tmem_base, cl);
        else if (p.bucket_hint)
            epilogue_rs_tma<true>(p, s, tmem_base, cl);
        else
            epilogue_rs_tma<false>(p, s, tmem_base, cl);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no cross-CTA traffic is left when either CTA releases TMEM
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}


cudaError_t prepare_one(int device, int *max_clusters) {
    // layouts: K-major / MN-major B, and both operands MN-major
    void (*fns[3])(KParams) = {cm_pair_kernel<0>, cm_pair_kernel<1>, cm_pair_kernel<3>};
    for (auto fn : fns) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmemBytes);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    int sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(unsigned(sms / CL * CL), 1, 1);
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, cm_pair_kernel<0>, &cfg);
    if (e != cudaSuccess) return e;
    *max_clusters = n;
    return cudaSuccess;
}

}  // namespace

int pair_rows() { return kPairRows; }

cudaError_t prepare_pair(int device, int *max_clusters) {
    static int cached[64] = {0};
    if (device < 0 || device >= 64) return cudaErrorInvalidValue;
    if (cached[device] == 0) {
        int n = 0;
        cudaError_t e = prepare_one(device, &n);
        if (e != cudaSuccess) return e;
        cached[device] = n > 0 ? n : -1;
    }
    *max_clusters = cached[device] > 0 ? cached[device] : 0;
    return cudaSuccess;
}

cudaError_t launch_pair(const KParams &p, int layout, int clusters, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(CL * clusters), 1, 1);
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (layout) {
        case 0: return cudaLaunchKernelEx(&cfg, cm_pair_kernel<0>, p);
        case 1: return cudaLaunchKernelEx(&cfg, cm_pair_kernel<1>, p);
        case 3: return cudaLaunchKernelEx(&cfg, cm_pair_kernel<3>, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace cm
