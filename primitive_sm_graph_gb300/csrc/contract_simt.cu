// float32 (and any-layout bf16) MUL+SUM contraction on the FP32 pipes.
//
// The tiled-matmul shape of limn's cuda device ("Backends": a block per
// output tile, both operands staged through shared memory, a patch of cells
// per thread in registers, the reduce axis walked in order).  Block tile
// 128x128, K slices of 16 (a short K, the case this kernel serves, takes
// few waits for its loads), 256 threads with an 8x8 register patch each;
// the View's strides are honoured for any layout.  Each output is one float32
// total over k in ascending order (multiply-adds may contract into FMA; the
// result is bounded by the reduction-order term like any SUM).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "contract.h"
#include "launch_util.cuh"

namespace psg {

namespace {

constexpr int TM = 128, TN = 128, TK = 16, NT = 256;

template <int DT>
__device__ __forceinline__ float ld(const void* p, int64_t o)
{
    if constexpr (DT == PSG_F32) return __ldg((const float*)p + o);
    else if constexpr (DT == PSG_F16) return __half2float(__ldg((const __half*)p + o));
    else return __uint_as_float(((uint32_t)__ldg((const unsigned short*)p + o)) << 16);
}

template <int DT>
__global__ void __launch_bounds__(NT) simt_gemm(const __grid_constant__ SimtParams p)
{
    pdl_enter();
    __shared__ float As[TK][TM + 4];
    __shared__ float Bs[TK][TN + 4];
    const int t = threadIdx.x;
    const int tx = t & 15, ty = t >> 4;
    const int64_t m0 = (int64_t)blockIdx.y * TM, n0 = (int64_t)blockIdx.x * TN;
    for (int64_t b = blockIdx.z; b < p.batch; b += gridDim.z) {
        const int64_t ab = p.a_off + b * p.a_bs, bb = p.b_off + b * p.b_bs;
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
        for (int64_t k0 = 0; k0 < p.K; k0 += TK) {
            // A slice [TM x TK]: with k stride 1 consecutive threads walk k
#pragma unroll
            for (int r = 0; r < TM * TK / NT; ++r) {
                const int idx = t + r * NT;
                int mm, kk;
                if (p.a_ks == 1) { mm = idx / TK; kk = idx % TK; } else { kk = idx / TM; mm = idx % TM; }
                const int64_t m = m0 + mm, k = k0 + kk;
                As[kk][mm] = (m < p.M && k < p.K) ? ld<DT>(p.A, ab + m * p.a_ms + k * p.a_ks) : 0.0f;
            }
#pragma unroll
            for (int r = 0; r < TN * TK / NT; ++r) {
                const int idx = t + r * NT;
                int nn, kk;
                if (p.b_ks == 1) { nn = idx / TK; kk = idx % TK; } else { kk = idx / TN; nn = idx % TN; }
                const int64_t n = n0 + nn, k = k0 + kk;
                Bs[kk][nn] = (n < p.N && k < p.K) ? ld<DT>(p.B, bb + n * p.b_ns + k * p.b_ks) : 0.0f;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < TK; ++kk) {
                float a[8], c[8];
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
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int64_t n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
                if (n >= p.N) continue;
                const int64_t o = p.c_off + b * p.c_bs + m * p.c_ms + n * p.c_ns;
                if (p.c_dtype == PSG_F32) ((float*)p.C)[o] = acc[i][j];
                else if (p.c_dtype == PSG_F16) ((__half*)p.C)[o] = __float2half_rn(acc[i][j]);
                else ((__nv_bfloat16*)p.C)[o] = __float2bfloat16_rn(acc[i][j]);
            }
        }
    }
}

dim3 grid_of(const SimtParams& p)
{
    const int64_t gz = p.batch < 65535 ? p.batch : 65535;
    return dim3((unsigned)((p.N + TN - 1) / TN), (unsigned)((p.M + TM - 1) / TM), (unsigned)gz);
}

}  // namespace

psg_status launch_contract_simt(const SimtParams& p, void* stream)
{
    if (p.M == 0 || p.N == 0 || p.batch == 0) return PSG_OK;
    if ((p.N + TN - 1) / TN > 2147483647 || (p.M + TM - 1) / TM > 65535) return PSG_E_UNSUPPORTED_LAYOUT;
    cudaStream_t s = (cudaStream_t)stream;
    if (p.ab_dtype == PSG_F32) launch(simt_gemm<PSG_F32>, grid_of(p), NT, 0, s, p);
    else if (p.ab_dtype == PSG_F16) launch(simt_gemm<PSG_F16>, grid_of(p), NT, 0, s, p);
    else launch(simt_gemm<PSG_BF16>, grid_of(p), NT, 0, s, p);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

void query_contract_simt(const SimtParams& p, int* grid, int* block, int* smem, int* regs)
{
    const dim3 g = grid_of(p);
    *grid = (int)(g.x * g.y * g.z);
    *block = NT;
    *smem = 0;
    *regs = kernel_regs(p.ab_dtype == PSG_F32   ? (const void*)simt_gemm<PSG_F32>
                        : p.ab_dtype == PSG_F16 ? (const void*)simt_gemm<PSG_F16>
                                                : (const void*)simt_gemm<PSG_BF16>);
}

}  // namespace psg
