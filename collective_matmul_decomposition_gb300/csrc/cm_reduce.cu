// cm_reduce.cu -- the reduction step of the pipelined GEMM -> ReduceScatter.
//
// "Hiding Tensor-Parallel Collectives: AG/RS Overlap in Megatron", section 6
// (pipeline chunks): the GEMM produces its output in c chunks and the
// ReduceScatter of chunk j runs while the GEMM computes chunk j + 1.  Here
// every logical rank r has written its fp32 partial product P_r for chunk j
// of every bucket o into the workspace; this kernel forms owner o's rows of
// that chunk, Y_o[j] = sum over r = 0 .. N-1 (in that order) of P_r[o][j],
// and rounds it into the output.  It is HBM-bound: N fp32 reads per output
// element, coalesced (consecutive threads take consecutive 16-byte groups of
// a row), with a grid-stride loop over every owner's chunk rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "cm_kernel.cuh"

namespace cm {
namespace {

constexpr int kReduceThreads = 256;

// P: partial buffers [N*N][Mb][n] fp32, buffer r*N + o = rank r's rows of
// bucket o.  y: [N][Mb][n].  Chunk j covers rows [j*rc, (j+1)*rc) of every
// bucket.  n4 = n / 4.
__global__ void __launch_bounds__(kReduceThreads) cm_reduce_chunk_kernel(const float4 *__restrict__ P, void *y, int N,
                                                                          int64_t Mb, int64_t rc, int64_t n4, int j,
                                                                          int y_f32) {
    const int64_t per_owner = rc * n4;
    const int64_t total = int64_t(N) * per_owner;
    const int64_t buf4 = Mb * n4;   // float4 groups per partial buffer
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const int o = int(idx / per_owner);
        const int64_t off = int64_t(j) * rc * n4 + (idx - int64_t(o) * per_owner);   // within the bucket
        float4 acc = __ldcs(P + int64_t(o) * buf4 + off);                          // rank 0
        for (int r = 1; r < N; ++r) {
            const float4 v = __ldcs(P + (int64_t(r) * N + o) * buf4 + off);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const int64_t yo = int64_t(o) * buf4 + off;   // 4-element group of y [N][Mb][n]
        if (y_f32) {
            reinterpret_cast<float4 *>(y)[yo] = acc;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t *>(&lo);
            u.y = *reinterpret_cast<uint32_t *>(&hi);
            reinterpret_cast<uint2 *>(y)[yo] = u;
        }
    }
}

}  // namespace

cudaError_t launch_reduce_chunk(const float *P, void *y, int N, int64_t Mb, int64_t rc, int64_t n, int j, bool y_f32,
                                int sms, cudaStream_t stream) {
    const int64_t total = int64_t(N) * rc * (n / 4);
    int64_t blocks = (total + kReduceThreads - 1) / kReduceThreads;
    blocks = blocks < int64_t(4) * sms ? blocks : int64_t(4) * sms;
    if (blocks < 1) return cudaSuccess;
    cm_reduce_chunk_kernel<<<unsigned(blocks), kReduceThreads, 0, stream>>>(
        reinterpret_cast<const float4 *>(P), y, N, Mb, rc, n / 4, j, y_f32 ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace cm
