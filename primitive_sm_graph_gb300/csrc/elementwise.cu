// Fused elementwise chain over Views (sm_103a).
//
// limn ("Backends") runs one thread per output cell.  Here one thread owns a
// chunk of VEC = 8 consecutive cells along the innermost dim: contiguous
// operands move with 128-bit loads and stores, a stride-0 (expanded) operand
// is read once per chunk, and the View's index arithmetic is per row (one
// multi-index decomposition per row, then col * inner_stride).  A block is
// split into row groups of a power-of-two size so short rows still fill the
// block; the grid is persistent (a multiple of the SM count) and strides over
// rows.
#include <cuda_runtime.h>

#include "interp.cuh"
#include "launch_util.cuh"

namespace psg {

namespace {

constexpr int EW_THREADS = 256;

template <int NIN>
struct EwSrc {
    uint32_t iv[NIN][VEC];
    template <int K>
    __device__ __forceinline__ uint32_t in(int v) const
    {
        if constexpr (K < NIN) return iv[K][v];
        else return 0u;
    }
    __device__ __forceinline__ uint32_t red(int) const { return 0u; }
};

// Load one operand's chunk into 32-bit value lanes.
__device__ __forceinline__ void load_chunk(const Operand& op, int64_t roff, bool rok, int64_t col0,
                                           int nvalid, uint32_t (&dst)[VEC])
{
    const int dt = op.dtype;
    switch (op.mode) {
    case IN_UNIFORM:
        dst[0] = load_cell(op.ptr, roff, dt);
        break;
    case IN_CONTIG: {
        const int64_t base = roff + col0;
        const int es = dt == PSG_F32 || dt == PSG_I32 ? 4 : dt == PSG_I8 ? 1 : 2;
        const char* p = (const char*)op.ptr + base * es;
        const bool full = nvalid == VEC;
        if (full && es == 4 && ((uintptr_t)p & 15) == 0) {
            uint4 a = __ldg((const uint4*)p), b = __ldg((const uint4*)p + 1);
            dst[0] = a.x; dst[1] = a.y; dst[2] = a.z; dst[3] = a.w;
            dst[4] = b.x; dst[5] = b.y; dst[6] = b.z; dst[7] = b.w;
        } else if (full && es == 2 && ((uintptr_t)p & 15) == 0) {
            uint4 a = __ldg((const uint4*)p);
            uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                uint32_t lo = w[v] & 0xffffu, hi = w[v] >> 16;
                if (dt == PSG_BF16) {
                    dst[2 * v] = lo << 16;
                    dst[2 * v + 1] = hi << 16;
                } else if (dt == PSG_F16) {
                    dst[2 * v] = f2u(__half2float(__ushort_as_half((unsigned short)lo)));
                    dst[2 * v + 1] = f2u(__half2float(__ushort_as_half((unsigned short)hi)));
                } else {
                    dst[2 * v] = (uint32_t)(int32_t)(int16_t)(uint16_t)lo;
                    dst[2 * v + 1] = (uint32_t)(int32_t)(int16_t)(uint16_t)hi;
                }
            }
        } else if (full && es == 1 && ((uintptr_t)p & 7) == 0) {
            uint2 a = __ldg((const uint2*)p);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                dst[v] = (uint32_t)(int32_t)(int8_t)(uint8_t)((a.x >> (8 * v)) & 0xffu);
                dst[4 + v] = (uint32_t)(int32_t)(int8_t)(uint8_t)((a.y >> (8 * v)) & 0xffu);
            }
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) dst[v] = v < nvalid ? load_cell(op.ptr, base + v, dt) : 0u;
        }
        break;
    }
    case IN_STRIDED:
#pragma unroll
        for (int v = 0; v < VEC; ++v)
            dst[v] = v < nvalid ? load_cell(op.ptr, roff + (col0 + v) * op.inner_stride, dt) : 0u;
        break;
    default: {  // IN_MASKED: the inner dim's mask is the last entry
        const int64_t lo = op.mlo[MAXD - 1], hi = op.mhi[MAXD - 1];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const int64_t c = col0 + v;
            const bool ok = rok && v < nvalid && c >= lo && c < hi;
            dst[v] = ok ? load_cell(op.ptr, roff + c * op.inner_stride, dt) : 0u;
        }
        break;
    }
    }
}

__device__ __forceinline__ void store_chunk(const Operand& op, int64_t roff, int64_t col0, int nvalid,
                                            const uint32_t (&val)[VEC])
{
    const int dt = op.dtype;
    if (op.inner_stride == 1 && nvalid == VEC) {
        const int64_t base = roff + col0;
        if (dt == PSG_F32 || dt == PSG_I32) {
            uint32_t* p = (uint32_t*)op.ptr + base;
            if (((uintptr_t)p & 15) == 0) {
                ((uint4*)p)[0] = make_uint4(val[0], val[1], val[2], val[3]);
                ((uint4*)p)[1] = make_uint4(val[4], val[5], val[6], val[7]);
                return;
            }
        } else if (dt == PSG_BF16 || dt == PSG_F16 || dt == PSG_I16) {
            unsigned short* p = (unsigned short*)op.ptr + base;
            if (((uintptr_t)p & 15) == 0) {
                uint32_t w[4];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint32_t lo, hi;
                    if (dt == PSG_BF16) { lo = val[2 * v] >> 16; hi = val[2 * v + 1] >> 16; }
                    else if (dt == PSG_F16) {
                        lo = __half_as_ushort(__float2half_rn(u2f(val[2 * v])));
                        hi = __half_as_ushort(__float2half_rn(u2f(val[2 * v + 1])));
                    } else { lo = val[2 * v] & 0xffffu; hi = val[2 * v + 1] & 0xffffu; }
                    w[v] = lo | (hi << 16);
                }
                *(uint4*)p = make_uint4(w[0], w[1], w[2], w[3]);
                return;
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) store_cell(const_cast<void*>(op.ptr), base + v, dt, val[v]);
        return;
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v)
        if (v < nvalid) store_cell(const_cast<void*>(op.ptr), roff + (col0 + v) * op.inner_stride, dt, val[v]);
}

template <int NIN>
__global__ void __launch_bounds__(EW_THREADS) ew_kernel(const __grid_constant__ EwLaunch L,
                                                        int group_log2)
{
    const int gs = 1 << group_log2;               // threads per row group
    const int groups = EW_THREADS >> group_log2;  // rows per block iteration
    const int grp = threadIdx.x >> group_log2;
    const int lane = threadIdx.x & (gs - 1);
    const int nd = L.sp.nd;
    const int n_in = L.n_in;
    for (int64_t row = (int64_t)blockIdx.x * groups + grp; row < L.sp.rows;
         row += (int64_t)gridDim.x * groups) {
        // per-row offsets: decompose the row into outer indices
        int64_t roff[NIN];
        bool rok[NIN];
#pragma unroll
        for (int k = 0; k < NIN; ++k) {
            roff[k] = k < n_in ? L.in[k].offset : 0;
            rok[k] = true;
        }
        int64_t ooff = L.out.offset;
        int64_t rem = row;
        for (int d = nd - 2; d >= 0; --d) {
            int64_t i;
            if (d > 0) {
                const int64_t s = L.sp.shape[d];
                const int64_t q = rem / s;
                i = rem - q * s;
                rem = q;
            } else {
                i = rem;
            }
            ooff += i * L.out.outer_stride[d];
#pragma unroll
            for (int k = 0; k < NIN; ++k) {
                if (k < n_in) {
                    roff[k] += i * L.in[k].outer_stride[d];
                    if (L.in[k].mode == IN_MASKED)
                        rok[k] = rok[k] && i >= L.in[k].mlo[d] && i < L.in[k].mhi[d];
                }
            }
        }
        for (int64_t ch = lane; ch < L.sp.chunks; ch += gs) {
            const int64_t col0 = ch * VEC;
            const int64_t left = L.sp.inner - col0;
            const int nvalid = left < VEC ? (int)left : VEC;
            EwSrc<NIN> src;
#pragma unroll
            for (int k = 0; k < NIN; ++k)
                if (k < n_in) load_chunk(L.in[k], roff[k], rok[k], col0, nvalid, src.iv[k]);
            RegFile r;
            run_program(L.prog.ins, L.prog.n, r, src);
            uint32_t res[VEC];
            result_vec(r, L.prog.out_reg, res);
            store_chunk(L.out, ooff, col0, nvalid, res);
        }
    }
}

int group_log2_for(int64_t chunks)
{
    int g = 0;
    while ((1 << g) < chunks && (1 << g) < EW_THREADS) ++g;
    return g;
}

}  // namespace

static void pick_launch(const EwLaunch& L, int* grid, int* lg, const void** fn)
{
    const int g = group_log2_for(L.sp.chunks);
    const int groups = EW_THREADS >> g;
    const int64_t need = (L.sp.rows + groups - 1) / groups;
    const void* f = L.n_in <= 4 ? (const void*)ew_kernel<4> : (const void*)ew_kernel<8>;
    const int per_sm = max_blocks_per_sm(f, EW_THREADS, 0);
    const int64_t cap = (int64_t)num_sms() * per_sm;
    *grid = (int)std::max<int64_t>(1, std::min<int64_t>(need, cap));
    *lg = g;
    *fn = f;
}

psg_status launch_elementwise(const EwLaunch& L, void* stream)
{
    if (L.sp.rows == 0 || L.sp.inner == 0) return PSG_OK;
    int grid, lg;
    const void* fn;
    pick_launch(L, &grid, &lg, &fn);
    cudaStream_t s = (cudaStream_t)stream;
    if (L.n_in <= 4) ew_kernel<4><<<grid, EW_THREADS, 0, s>>>(L, lg);
    else ew_kernel<8><<<grid, EW_THREADS, 0, s>>>(L, lg);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

void query_elementwise(const EwLaunch* L, int* grid, int* block, int* smem, int* regs)
{
    int g, lg;
    const void* fn;
    pick_launch(*L, &g, &lg, &fn);
    *grid = g;
    *block = EW_THREADS;
    *smem = 0;
    *regs = kernel_regs(fn);
}

}  // namespace psg
