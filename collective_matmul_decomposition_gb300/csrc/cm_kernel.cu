// cm_kernel.cu -- the persistent tile kernel that runs a plan's task table.
//
// Every task is one partial GEMM of the decomposition ("Overlap
// Communication with Dependent Computation via Decomposition in Large Deep
// Learning Models", section "The idea"): A rows [rows_c per chunk, K] of the
// shard or slab the task names, times B = W_r, over 128 x 256 output tiles.
// Tiles of all tasks form one linear sequence (task-major, then chunk, then
// row tile, then column tile) that CTA b walks as b, b + grid, b + 2*grid...
//
// Roles inside a CTA (256 threads, one CTA per SM):
//   warp 0  TMA producer: waits until the task's input chunk is resident
//           (AG: the forward that filled the slot), then streams A and B
//           K-slices into a 4-stage shared-memory ring.
//   warp 1  MMA issuer: tcgen05.mma 128x256x16 into one of two TMEM
//           accumulators; commits free ring stages and full accumulators.
//           AG: after the last K-slice of a tile has landed it counts the
//           slot's rows as read (the slot may then be overwritten).
//   warp 2  AG forwarder: for the first column tile of each row tile it
//           TMA-stores every landed A slice into the ring neighbour's receive
//           slot -- the shard is forwarded while it is being multiplied, the
//           way the pages pair each partial product with a transfer -- and
//           releases the slot's ready flag once the stores are complete.
//   warps 4-7 epilogue: TMEM -> registers; AG writes the tile into the
//           shard's rows of Y_r (the DynamicUpdateSlice); RS adds the received
//           fp32 partial bucket(s) and writes the sum to the next rank's
//           receive buffer, or rounds it into the output at the owner.
//
// Every wait (mbarrier or cross-CTA flag) is bounded by p.timeout_ns; on
// expiry the first failing thread records {code, task, chunk, site} in the
// status word, the CTA stops issuing work, waits for its own copies in
// flight, releases TMEM and exits.
#include <cuda_bf16.h>

#include "cm_kernel_common.cuh"

namespace cm {
namespace {

using namespace dev;
using namespace kc;

struct Smem {
    uint8_t *a[kStages];
    uint8_t *b[kStages];
    uint64_t *full, *empty, *tfull, *tempty, *drain;
    uint32_t *tmem_slot;
    volatile int *abort;
};

template <bool B_MN>
__device__ void producer(const KParams &p, const Smem &s, int total) {
    int stage = 0;
    uint32_t phase = 0;
    int last_parity[kStages];
    for (int i = 0; i < kStages; ++i) last_parity[i] = -1;
    const uint32_t tx = uint32_t(p.a_box_rows) * kBK * 2 + kBBytes;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
        if (*s.abort) break;
        const TileCoord c = decode(p, t);
        if (!in_bounds(p, c.task >= p.task_begin && c.task < p.task_end && c.q >= 0 && c.q < p.chunks,
                       kSiteBoundsTask, c.task, c.q))
            break;
        const cm_task &tk = p.tasks[c.task];
        if (p.op == 0 && tk.wait_in[0] >= 0) {
            if (!wait_flag(p, s.abort, flag_ptr(p, tk.wait_in[0], c.q, c.mt, 0), p.tgt_in, kSiteProducerFlag, c.task, c.q)) break;
            fence_proxy_async_global();
        }
        const void *tmA = tk.a_src == 1 ? static_cast<const void *>(&p.tmA1) : static_cast<const void *>(&p.tmA0);
        const int row0 = c.mt * kBM, n0 = c.nt * kBN;
        const int nk = kslices(p, tk);
        bool ok = true;
        for (int kk = 0; kk < nk; ++kk) {
            int rr = tk.rank, kb = kk, slab = tk.a_slab * p.chunks + c.q;
            if (tk.a_src == 2) {
                rr = kk / p.kblocks;
                kb = kk - rr * p.kblocks;
                slab = (rr * p.N + tk.out_idx) * p.chunks + c.q;
            }
            if (!wait_mbar<false>(p, s.abort, &s.empty[stage], phase ^ 1u, kSiteEmpty, c.task, c.q)) {
                ok = false;
                break;
            }
            mbar_expect_tx(&s.full[stage], tx);
            tma_load_3d(s.a[stage], tmA, &s.full[stage], kb * kBK, row0, slab);
            if (B_MN) {
                for (int j = 0; j < kBN / 64; ++j)
                    tma_load_3d(s.b[stage] + j * (64 * kBK * 2), &p.tmB, &s.full[stage], n0 + 64 * j, kb * kBK, rr);
            } else {
                tma_load_3d(s.b[stage], &p.tmB, &s.full[stage], kb * kBK, n0, rr);
            }
            last_parity[stage] = int(phase);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
    }
    // no CTA may exit with a TMA load still writing its shared memory
    for (int i = 0; i < kStages; ++i)
        if (last_parity[i] >= 0) drain_mbar<false>(p, &s.full[i], uint32_t(last_parity[i]));
}

template <bool B_MN>
__device__ void mma_issuer(const KParams &p, const Smem &s, int total, uint32_t tmem_base) {
    constexpr uint32_t kIdesc = idesc_bf16(kBM, kBN, B_MN);
    // K-major SW128 (A, and B when K-major): rows of 128 B, 8-row groups 1024 B apart;
    // one K=16 step is 32 B along the row.
    // n-major SW128 B: 64-column blocks 8 KB apart (leading offset), 8-row
    // K groups 1024 B apart (stride offset); one K=16 step is 16 rows = 2 KB.
    constexpr uint32_t kBLbo = B_MN ? 64 * kBK * 2 : 16;
    constexpr uint32_t kBStep = B_MN ? (16 * 128) >> 4 : 32 >> 4;
    int stage = 0;
    uint32_t phase = 0;
    int accb = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
        if (*s.abort) break;
        const TileCoord c = decode(p, t);
        const cm_task &tk = p.tasks[c.task];
        if (!wait_mbar<false>(p, s.abort, &s.tempty[accb], acc_phase ^ 1u, kSiteTmemEmpty, c.task, c.q)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(accb * kBN);
        const int nk = kslices(p, tk);
        bool ok = true;
        for (int kk = 0; kk < nk; ++kk) {
            if (!wait_mbar<false>(p, s.abort, &s.full[stage], phase, kSiteFull, c.task, c.q)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t ad = desc_sw128(smem_u32(s.a[stage]), 16, 1024);
            const uint64_t bd = desc_sw128(smem_u32(s.b[stage]), kBLbo, 1024);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
                mma_bf16(d, ad + uint64_t(2 * k), bd + uint64_t(kBStep * k), kIdesc, (kk | k) != 0 ? 1u : 0u);
            mma_commit(&s.empty[stage]);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        mma_commit(&s.tfull[accb]);
        // AG: every K slice of this tile's A rows has landed in shared memory,
        // so the slot rows it read may be overwritten by the next forward.
        if (p.op == 0 && tk.sig_done >= 0) red_release_add(flag_ptr(p, tk.sig_done, c.q, c.mt, 0), 1u);
        if (++accb == 2) {
            accb = 0;
            acc_phase ^= 1u;
        }
    }
    // every MMA this thread issued must finish before TMEM is released
    mma_commit(s.drain);
    drain_mbar<false>(p, s.drain, 0);
}

__device__ void forwarder(const KParams &p, const Smem &s, int total) {
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
        if (*s.abort) break;
        const TileCoord c = decode(p, t);
        const cm_task &tk = p.tasks[c.task];
        const bool fwd = c.nt == 0 && (tk.fwd_slot[0] >= 0 || tk.fwd_slot[1] >= 0);
        bool ok = true;
        if (fwd) {
            for (int j = 0; j < 2 && ok; ++j)
                if (tk.fwd_slot[j] >= 0 && tk.wait_free[j] >= 0)
                    ok = wait_flag(p, s.abort, flag_ptr(p, tk.wait_free[j], c.q, c.mt, 0), p.tgt_free, kSiteForwardFlag, c.task, c.q);
            if (!ok) break;
            fence_proxy_async_global();
        }
        const int nk = kslices(p, tk);
        int pending = -1;
        for (int kk = 0; kk < nk; ++kk) {
            if (!wait_mbar<false>(p, s.abort, &s.full[stage], phase, kSiteForwardFull, c.task, c.q)) {
                ok = false;
                break;
            }
            if (fwd) {
                for (int j = 0; j < 2; ++j)
                    if (tk.fwd_slot[j] >= 0)
                        tma_store_3d(&p.tmA1, s.a[stage], kk * kBK, c.mt * kBM, tk.fwd_slot[j] * p.chunks + c.q);
                bulk_commit();
                if (pending >= 0) {   // the previous slice's stores have read shared memory
                    bulk_wait_read<1>();
                    mbar_arrive(&s.empty[pending]);
                }
                pending = stage;
            } else {
                mbar_arrive(&s.empty[stage]);
            }
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        if (fwd) {
            bulk_wait_read<0>();
            if (pending >= 0) mbar_arrive(&s.empty[pending]);
            bulk_wait<0>();               // the stores are complete in global memory
            fence_proxy_async_global();
            for (int j = 0; j < 2; ++j)
                if (tk.fwd_slot[j] >= 0 && tk.sig_fwd[j] >= 0) red_release_add(flag_ptr(p, tk.sig_fwd[j], c.q, c.mt, 0), 1u);
        }
    }
    bulk_wait<0>();
}

__device__ void epilogue(const KParams &p, const Smem &s, int total, uint32_t tmem_base) {
    const int et = int(threadIdx.x) - 128;   // 0..127 = row of the tile
    const int ew = et >> 5;                   // warp 4..7 reads TMEM lanes 32*(warp%4)..
    int accb = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const TileCoord c = decode(p, t);
        const cm_task &tk = p.tasks[c.task];
        bool bad = !wait_mbar<false>(p, s.abort, &s.tfull[accb], acc_phase, kSiteTmemFull, c.task, c.q);
        if (p.op == 1 && et == 0 && !bad) {
            for (int j = 0; j < 2 && !bad; ++j)
                if (tk.wait_in[j] >= 0)
                    bad = !wait_flag(p, s.abort, flag_ptr(p, tk.wait_in[j], c.q, c.mt, c.nt), p.tgt_in, kSiteEpilogueFlag, c.task, c.q);
            if (!bad && tk.wait_free[0] >= 0)
                bad = !wait_flag(p, s.abort, flag_ptr(p, tk.wait_free[0], c.q, c.mt, c.nt), p.tgt_free, kSiteEpilogueFlag, c.task, c.q);
        }
        bad = bar_or(1, 128, bad || *s.abort != 0);
        if (bad) break;
        tc_fence_after();

        const int row = c.mt * kBM + et;          // row inside the chunk
        const int64_t crow = int64_t(c.q) * p.rows_c + row;   // row inside the shard / bucket
        bool row_ok = row < p.rows_c;
        if (kCheckBounds && row_ok) {   // debug builds: every global row this thread touches
            const int64_t yrow = (p.op == 0 ? int64_t(tk.rank) * (p.y_rank_stride / p.n) : 0) +
                                 int64_t(tk.out_idx) * p.out_rows_per_idx + crow;
            const bool y_ok = (yrow + 1) * p.n <= p.y_elems;
            const bool okb = p.op == 0 ? y_ok
                                       : tk.out_buf < p.acc_bufs && tk.in_buf[0] < p.acc_bufs &&
                                             tk.in_buf[1] < p.acc_bufs && (tk.out_buf >= 0 || y_ok);
            row_ok = in_bounds(p, okb, p.op == 0 ? kSiteBoundsOutput : kSiteBoundsBucket, c.task, c.q);
        }
        for (int cb = 0; cb < kBN / 32; ++cb) {
            uint32_t v[32];
            tmem_ld32(tmem_base + (uint32_t(ew * 32) << 16) + uint32_t(accb * kBN + cb * 32), v);
            tmem_wait_ld();
            const int col0 = c.nt * kBN + cb * 32;
            if (!row_ok || col0 >= p.n) continue;
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
            int64_t orow;   // element offset of (row, col0) in the destination
            bool to_acc = false;
            if (p.op == 0) {
                orow = int64_t(tk.rank) * p.y_rank_stride + (int64_t(tk.out_idx) * p.out_rows_per_idx + crow) * p.n;
            } else {
                const int64_t brow = crow * p.n;
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (tk.in_buf[j] >= 0) {
                        const float4 *src =
                            reinterpret_cast<const float4 *>(p.acc + int64_t(tk.in_buf[j]) * p.acc_buf_stride + brow + col0);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (col0 + 4 * i < p.n) add4(f + 4 * i, __ldcg(src + i));
                    }
                if (tk.out_buf >= 0) {
                    to_acc = true;
                    orow = int64_t(tk.out_buf) * p.acc_buf_stride + brow;
                } else {
                    orow = (int64_t(tk.out_idx) * p.out_rows_per_idx + crow) * p.n;
                }
            }
            if (to_acc) {
                float4 *dst = reinterpret_cast<float4 *>(p.acc + orow + col0);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (col0 + 4 * i < p.n) dst[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
            } else if (p.y_f32) {
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
        tc_fence_before();
        mbar_arrive(&s.tempty[accb]);
        if (p.op == 1 && tk.sig_done >= 0) {
            __threadfence();
            bar_sync(1, 128);
            if (et == 0) red_release_add(flag_ptr(p, tk.sig_done, c.q, c.mt, c.nt), 1u);
        }
        if (++accb == 2) {
            accb = 0;
            acc_phase ^= 1u;
        }
    }
}

template <bool B_MN>
__global__ void __launch_bounds__(kThreads, 1) cm_persistent_kernel(const __grid_constant__ KParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem s;
    for (int i = 0; i < kStages; ++i) {
        s.a[i] = base + i * kABytes;
        s.b[i] = base + kStages * kABytes + i * kBBytes;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + kStages * (kABytes + kBBytes));
    s.full = bars;
    s.empty = bars + kStages;
    s.tfull = bars + 2 * kStages;
    s.tempty = bars + 2 * kStages + 2;
    s.drain = bars + 2 * kStages + 4;
    s.tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kStages + 5);
    s.abort = reinterpret_cast<volatile int *>(bars + 2 * kStages + 6);

    const int warp = int(threadIdx.x) >> 5, lane = int(threadIdx.x) & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], p.op == 0 ? 2 : 1);   // AG: MMA commit + forwarder
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tfull[i], 1);
            mbar_init(&s.tempty[i], 128);
        }
        mbar_init(s.drain, 1);
        *s.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&p.tmA0);
        prefetch_tmap(&p.tmA1);
        prefetch_tmap(&p.tmB);
    }
    if (warp == 1) {
        tmem_alloc(s.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s.tmem_slot;
    const int total = (p.task_end - p.task_begin) * p.tiles_per_task;

    if (warp == 0) {
        if (lane == 0) producer<B_MN>(p, s, total);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) mma_issuer<B_MN>(p, s, total, tmem_base);
        __syncwarp();
    } else if (warp == 2) {
        if (lane == 0 && p.op == 0) forwarder(p, s, total);
        __syncwarp();
    } else if (warp >= 4) {
        epilogue(p, s, total, tmem_base);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

cudaError_t prepare_device(int device, int *num_sms) {
    static int sms[64] = {0};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (sms[device] == 0) {
        cudaError_t e = cudaFuncSetAttribute(cm_persistent_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(cm_persistent_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        int v = 0;
        e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device);
        if (e != cudaSuccess) return e;
        sms[device] = v;
    }
    *num_sms = sms[device];
    return cudaSuccess;
}

cudaError_t launch_persistent(const KParams &p, bool b_mn_major, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs co-resident: flag waits cannot starve
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (b_mn_major) return cudaLaunchKernelEx(&cfg, cm_persistent_kernel<true>, p);
    return cudaLaunchKernelEx(&cfg, cm_persistent_kernel<false>, p);
}

}  // namespace cm
