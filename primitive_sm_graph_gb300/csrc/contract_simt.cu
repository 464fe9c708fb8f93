// MUL+SUM contraction on the FP32 / FP64 / integer pipes: float32 (short K),
// any-layout bf16 / f16, float64, the integer dtypes and masked (padded) Views.
//
// The tiled-matmul shape of limn's cuda device ("Backends": a block per
// output tile, both operands staged through shared memory, a patch of cells
// per thread in registers, the reduce axis walked in order).  Block tile
// 128x128, K slices of 16 (a short K, the case this kernel serves, takes
// few waits for its loads), 256 threads with an 8x8 register patch each;
// the View's strides are honoured for any layout.  Each output is one total
// over k in ascending order: float32 for the float dtypes up to 32 bits
// (multiply-adds may contract into FMA; the result is bounded by the
// reduction-order term like any SUM), float64 for float64, and uint32 with
// wraparound for the integers (limn, "Three rules hold it together": integer
// arithmetic wraps modulo 2^width), stored modulo the output's width.
//
// A masked operand reads zero outside its mask.  A's mask along m and k and
// B's along n and k are applied as the tiles load (the zero factors are
// multiplied in, as the broadcast product would); a mask across the other
// operand's broadcast axis (A's along n, B's along m, either along a batch
// dim) zeroes whole output cells, which are written 0.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "contract.h"
#include "launch_util.cuh"

namespace psg {

namespace {

constexpr int TM = 128, TN = 128, TK = 16, NT = 256;

// accumulator of an input dtype
template <int DT> struct AccOf { using T = float; };
template <> struct AccOf<PSG_F64> { using T = double; };
template <> struct AccOf<PSG_I32> { using T = uint32_t; };
template <> struct AccOf<PSG_I16> { using T = uint32_t; };
template <> struct AccOf<PSG_I8> { using T = uint32_t; };

template <int DT>
__device__ __forceinline__ typename AccOf<DT>::T ld(const void* p, int64_t o)
{
    if constexpr (DT == PSG_F32) return __ldg((const float*)p + o);
    else if constexpr (DT == PSG_F16) return __half2float(__ldg((const __half*)p + o));
    else if constexpr (DT == PSG_BF16) return __uint_as_float(((uint32_t)__ldg((const unsigned short*)p + o)) << 16);
    else if constexpr (DT == PSG_F64) return __ldg((const double*)p + o);
    else if constexpr (DT == PSG_I32) return (uint32_t)__ldg((const int*)p + o);
    else if constexpr (DT == PSG_I16) return (uint32_t)(int)__ldg((const short*)p + o);
    else return (uint32_t)(int)__ldg((const signed char*)p + o);
}

__device__ __forceinline__ void st(const SimtParams& p, int64_t o, float v)
{
    if (p.c_dtype == PSG_F32) ((float*)p.C)[o] = v;
    else if (p.c_dtype == PSG_F16) ((__half*)p.C)[o] = __float2half_rn(v);
    else ((__nv_bfloat16*)p.C)[o] = __float2bfloat16_rn(v);
}
__device__ __forceinline__ void st(const SimtParams& p, int64_t o, double v) { ((double*)p.C)[o] = v; }
__device__ __forceinline__ void st(const SimtParams& p, int64_t o, uint32_t v)
{
    if (p.c_dtype == PSG_I32) ((int32_t*)p.C)[o] = (int32_t)v;
    else if (p.c_dtype == PSG_I16) ((uint16_t*)p.C)[o] = (uint16_t)(v & 0xffffu);
    else ((uint8_t*)p.C)[o] = (uint8_t)(v & 0xffu);
}

// MASKED: the read windows and the cell window are applied; otherwise the
// operands are read in full (the windows are the whole shape) and the
// bounds are the tile edges alone
template <int DT, bool MASKED>
__global__ void __launch_bounds__(NT) simt_gemm(const __grid_constant__ SimtParams p)
{
    pdl_enter();
    using Acc = typename AccOf<DT>::T;
    __shared__ Acc As[TK][TM + 4];
    __shared__ Acc Bs[TK][TN + 4];
    const int t = threadIdx.x;
    const int tx = t & 15, ty = t >> 4;
    const int64_t m0 = (int64_t)blockIdx.y * TM, n0 = (int64_t)blockIdx.x * TN;
    for (int64_t b = blockIdx.z; b < p.batch; b += gridDim.z) {
        const int64_t ab = p.a_off + b * p.a_bs, bb = p.b_off + b * p.b_bs;
        Acc acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = Acc(0);
        for (int64_t k0 = 0; k0 < p.K; k0 += TK) {
            // A slice [TM x TK]: with k stride 1 consecutive threads walk k
#pragma unroll
            for (int r = 0; r < TM * TK / NT; ++r) {
                const int idx = t + r * NT;
                int mm, kk;
                if (p.a_ks == 1) { mm = idx / TK; kk = idx % TK; } else { kk = idx / TM; mm = idx % TM; }
                const int64_t m = m0 + mm, k = k0 + kk;
                As[kk][mm] = (MASKED ? (m >= p.a_mlo && m < p.a_mhi && k >= p.a_klo && k < p.a_khi) : (m < p.M && k < p.K))
                                 ? ld<DT>(p.A, ab + m * p.a_ms + k * p.a_ks)
                                 : Acc(0);
            }
#pragma unroll
            for (int r = 0; r < TN * TK / NT; ++r) {
                const int idx = t + r * NT;
                int nn, kk;
                if (p.b_ks == 1) { nn = idx / TK; kk = idx % TK; } else { kk = idx / TN; nn = idx % TN; }
                const int64_t n = n0 + nn, k = k0 + kk;
                Bs[kk][nn] = (MASKED ? (n >= p.b_nlo && n < p.b_nhi && k >= p.b_klo && k < p.b_khi) : (n < p.N && k < p.K))
                                 ? ld<DT>(p.B, bb + n * p.b_ns + k * p.b_ks)
                                 : Acc(0);
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < TK; ++kk) {
                Acc a[8], c[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    a[i] = As[kk][ty * 4 + i];
                    a[4 + i] = As[kk][64 + ty * 4 + i];
                    c[i] = Bs[kk][tx * 4 + i];
                    c[4 + i] = Bs[kk][64 + tx * 4 + i];
                }
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] += a[i] * c[j];
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
            if (m >= p.M) continue;
            const bool mk = !MASKED || (m >= p.c_mlo && m < p.c_mhi);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int64_t n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
                if (n >= p.N) continue;
                const bool keep = mk && (!MASKED || (n >= p.c_nlo && n < p.c_nhi));
                st(p, p.c_off + b * p.c_bs + m * p.c_ms + n * p.c_ns, keep ? acc[i][j] : Acc(0));
            }
        }
    }
}

dim3 grid_of(const SimtParams& p)
{
    const int64_t gz = p.batch < 65535 ? p.batch : 65535;
    return dim3((unsigned)((p.N + TN - 1) / TN), (unsigned)((p.M + TM - 1) / TM), (unsigned)gz);
}

// true when a window is narrower than the shape (a mask is in effect)
bool masked(const SimtParams& p)
{
    return p.a_mlo != 0 || p.a_mhi != p.M || p.a_klo != 0 || p.a_khi != p.K || p.b_nlo != 0 || p.b_nhi != p.N ||
           p.b_klo != 0 || p.b_khi != p.K || p.c_mlo != 0 || p.c_mhi != p.M || p.c_nlo != 0 || p.c_nhi != p.N;
}

template <bool MK>
const void* kernel_of(int dt)
{
    switch (dt) {
    case PSG_F32: return (const void*)simt_gemm<PSG_F32, MK>;
    case PSG_BF16: return (const void*)simt_gemm<PSG_BF16, MK>;
    case PSG_F16: return (const void*)simt_gemm<PSG_F16, MK>;
    case PSG_F64: return (const void*)simt_gemm<PSG_F64, MK>;
    case PSG_I32: return (const void*)simt_gemm<PSG_I32, MK>;
    case PSG_I16: return (const void*)simt_gemm<PSG_I16, MK>;
    case PSG_I8: return (const void*)simt_gemm<PSG_I8, MK>;
    }
    return nullptr;
}

template <bool MK>
psg_status launch_typed(const SimtParams& p, dim3 g, cudaStream_t s)
{
    switch (p.ab_dtype) {
    case PSG_F32: launch(simt_gemm<PSG_F32, MK>, g, NT, 0, s, p); break;
    case PSG_BF16: launch(simt_gemm<PSG_BF16, MK>, g, NT, 0, s, p); break;
    case PSG_F16: launch(simt_gemm<PSG_F16, MK>, g, NT, 0, s, p); break;
    case PSG_F64: launch(simt_gemm<PSG_F64, MK>, g, NT, 0, s, p); break;
    case PSG_I32: launch(simt_gemm<PSG_I32, MK>, g, NT, 0, s, p); break;
    case PSG_I16: launch(simt_gemm<PSG_I16, MK>, g, NT, 0, s, p); break;
    case PSG_I8: launch(simt_gemm<PSG_I8, MK>, g, NT, 0, s, p); break;
    default: return PSG_E_UNSUPPORTED_DTYPE;
    }
    return PSG_OK;
}

}  // namespace

psg_status launch_contract_simt(const SimtParams& p, void* stream)
{
    if (p.M == 0 || p.N == 0 || p.batch == 0) return PSG_OK;
    if ((p.N + TN - 1) / TN > 2147483647 || (p.M + TM - 1) / TM > 65535) return PSG_E_UNSUPPORTED_LAYOUT;
    cudaStream_t s = (cudaStream_t)stream;
    const psg_status st = masked(p) ? launch_typed<true>(p, grid_of(p), s) : launch_typed<false>(p, grid_of(p), s);
    if (st != PSG_OK) return st;
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

void query_contract_simt(const SimtParams& p, int* grid, int* block, int* smem, int* regs)
{
    const dim3 g = grid_of(p);
    *grid = (int)(g.x * g.y * g.z);
    *block = NT;
    *smem = 0;
    const void* f = masked(p) ? kernel_of<true>(p.ab_dtype) : kernel_of<false>(p.ab_dtype);
    *regs = f ? kernel_regs(f) : 0;
}

}  // namespace psg
