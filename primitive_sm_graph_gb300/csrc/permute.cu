// CONTIGUOUS of a permuted View: out[i] = in[perm(i)] (sm_103a).
//
// A permute is a View (limn, "Three rules hold it together") and copying it
// out is a cut (limn, "Reading the schedule").  When the input's stride-1 dim
// is not the output's stride-1 dim the copy is a transpose: both sides must
// stay coalesced, so a 64x64 tile is staged through shared memory (Tiki,
// "What works today": a shared-memory transpose).  The tile is padded by one
// element per row, so both the row-wise writes and the column-wise reads hit
// 32 distinct banks.  The grid is persistent over (batch, tile-row, tile-col).
#include <cuda_runtime.h>

#include "common.h"
#include "launch_util.cuh"
#include "permute.h"

namespace psg {

namespace {

constexpr int TT = 64;       // tile edge
constexpr int TX = 32;       // threads along the contiguous edge
constexpr int TY = 8;        // thread rows
constexpr int TTHREADS = TX * TY;

template <typename E>
__global__ void __launch_bounds__(TTHREADS) transpose_kernel(const __grid_constant__ TransposeLaunch L)
{
    pdl_enter();
    __shared__ E tile[TT][TT + 1];
    const E* __restrict__ src = (const E*)L.in;
    E* __restrict__ dst = (E*)L.out;
    const int tx = threadIdx.x % TX, ty = threadIdx.x / TX;
    const int64_t ta = (L.A + TT - 1) / TT, ti = (L.I + TT - 1) / TT;
    const int64_t per_batch = ta * ti;
    const int64_t total = per_batch * L.batch;
    for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
        const int64_t b = t / per_batch;
        const int64_t rr = t - b * per_batch;
        const int64_t ia = rr / ti, ii = rr - ia * ti;
        const int64_t a0 = ia * TT, i0 = ii * TT;
        // batch offsets
        int64_t in_off = L.in_offset, out_off = L.out_offset, rem = b;
        for (int d = L.nb - 1; d >= 0; --d) {
            const int64_t q = rem / L.bshape[d];
            const int64_t x = rem - q * L.bshape[d];
            rem = q;
            in_off += x * L.in_bstride[d];
            out_off += x * L.out_bstride[d];
        }
        // read: input rows run along i (stride in_si), each row is contiguous
        // in a; all loads are issued before the shared-memory stores
        E v[TT / TY][TT / TX];
#pragma unroll
        for (int k = 0; k < TT / TY; ++k) {
            const int64_t i = i0 + ty + k * TY;
#pragma unroll
            for (int q = 0; q < TT / TX; ++q) {
                const int64_t a = a0 + tx + q * TX;
                v[k][q] = (i < L.I && a < L.A) ? src[in_off + i * L.in_si + a] : E(0);
            }
        }
#pragma unroll
        for (int k = 0; k < TT / TY; ++k)
#pragma unroll
            for (int q = 0; q < TT / TX; ++q) tile[ty + k * TY][tx + q * TX] = v[k][q];
        __syncthreads();
        // write: output rows run along a (stride out_sa), each row contiguous in i
#pragma unroll
        for (int k = 0; k < TT / TY; ++k) {
            const int64_t a = a0 + ty + k * TY;
#pragma unroll
            for (int q = 0; q < TT / TX; ++q) {
                const int64_t i = i0 + tx + q * TX;
                if (i < L.I && a < L.A) dst[out_off + a * L.out_sa + i] = tile[tx + q * TX][ty + k * TY];
            }
        }
        __syncthreads();
    }
}

template <typename E>
void launch_t(const TransposeLaunch& L, cudaStream_t s)
{
    const int64_t tiles = L.batch * ((L.A + TT - 1) / TT) * ((L.I + TT - 1) / TT);
    const int per_sm = max_blocks_per_sm((const void*)transpose_kernel<E>, TTHREADS, 0);
    const int64_t cap = (int64_t)num_sms() * per_sm;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, cap));
    launch(transpose_kernel<E>, grid, TTHREADS, 0, s, L);
}

// Generic strided copy for layouts the tile does not cover (any dtype):
// one thread per output cell, the View's index arithmetic per cell.
__global__ void copy_kernel(const __grid_constant__ CopyLaunch L)
{
    pdl_enter();
    const int64_t n = L.numel;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        int64_t rem = e, ioff = L.in_offset, ooff = L.out_offset;
        bool ok = true;
        for (int d = L.nd - 1; d >= 0; --d) {
            const int64_t q = rem / L.shape[d];
            const int64_t x = rem - q * L.shape[d];
            rem = q;
            ioff += x * L.in_stride[d];
            ooff += x * L.out_stride[d];
            ok = ok && x >= L.mlo[d] && x < L.mhi[d];
        }
        const char* s = (const char*)L.in + ioff * L.es;
        char* o = (char*)L.out + ooff * L.es;
        switch (L.es) {
        case 1: *(uint8_t*)o = ok ? *(const uint8_t*)s : 0; break;
        case 2: *(uint16_t*)o = ok ? *(const uint16_t*)s : 0; break;
        case 4: *(uint32_t*)o = ok ? *(const uint32_t*)s : 0; break;
        default: *(uint64_t*)o = ok ? *(const uint64_t*)s : 0; break;
        }
    }
}

}  // namespace

psg_status launch_transpose(const TransposeLaunch& L, void* stream)
{
    if (L.A == 0 || L.I == 0 || L.batch == 0) return PSG_OK;
    cudaStream_t s = (cudaStream_t)stream;
    switch (L.es) {
    case 1: launch_t<uint8_t>(L, s); break;
    case 2: launch_t<uint16_t>(L, s); break;
    case 4: launch_t<uint32_t>(L, s); break;
    default: launch_t<uint64_t>(L, s); break;
    }
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

psg_status launch_copy(const CopyLaunch& L, void* stream)
{
    if (L.numel == 0) return PSG_OK;
    const int threads = 256;
    const int per_sm = max_blocks_per_sm((const void*)copy_kernel, threads, 0);
    const int64_t need = (L.numel + threads - 1) / threads;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)num_sms() * per_sm));
    launch(copy_kernel, grid, threads, 0, (cudaStream_t)stream, L);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

void query_transpose(int es, int64_t tiles, int* grid, int* block, int* smem, int* regs)
{
    const void* f = es == 1 ? (const void*)transpose_kernel<uint8_t>
                  : es == 2 ? (const void*)transpose_kernel<uint16_t>
                  : es == 4 ? (const void*)transpose_kernel<uint32_t>
                            : (const void*)transpose_kernel<uint64_t>;
    const int per_sm = max_blocks_per_sm(f, TTHREADS, 0);
    *grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)num_sms() * per_sm));
    *block = TTHREADS;
    *smem = 0;
    *regs = kernel_regs(f);
}

}  // namespace psg
