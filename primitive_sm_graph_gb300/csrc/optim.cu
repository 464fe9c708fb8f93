// AdamW step over a list of tensors in one launch (sm_103a).
//
// limn ("nn, optim and checkpoints": optimizer steps are ASSIGN graphs over
// the parameters, beta**t kept on the device) -- here the whole update of
// every tensor of the list is one elementwise launch over their concatenated
// index space, plus one single-thread launch that advances beta1^t, beta2^t.
// Per element, in float32, each operation rounded in this order (decoupled
// weight decay, Loshchilov & Hutter's AdamW in torch.optim.AdamW's order):
//   p1 = p * (1 - lr*wd)
//   m' = b1*m + (1-b1)*g          v' = b2*v + (1-b2)*(g*g)
//   denom = sqrt(v') / sqrt(1 - b2^t) + eps
//   p' = p1 - (lr / (1 - b1^t)) * (m' / denom)
// with b^t the running products after this step; p' rounds once into the
// parameter dtype.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "common.h"
#include "launch_util.cuh"

namespace psg {

namespace {

constexpr int GROUP = 32;  // tensors per launch

struct AdamWLaunch {
    void* p[GROUP];
    const void* g[GROUP];
    float* m[GROUP];
    float* v[GROUP];
    long long start[GROUP + 1];   // prefix offsets of the concatenated index space
    int count;
    int dtype;
    float lr, b1, b2, eps, wd;
    const float* bpow;            // beta1^t, beta2^t before this step
};

template <int DT>
__device__ __forceinline__ float ldp(const void* p, long long i)
{
    if constexpr (DT == PSG_F32) return ((const float*)p)[i];
    else if constexpr (DT == PSG_BF16) return __bfloat162float(((const __nv_bfloat16*)p)[i]);
    else return __half2float(((const __half*)p)[i]);
}
template <int DT>
__device__ __forceinline__ void stp(void* p, long long i, float x)
{
    if constexpr (DT == PSG_F32) ((float*)p)[i] = x;
    else if constexpr (DT == PSG_BF16) ((__nv_bfloat16*)p)[i] = __float2bfloat16_rn(x);
    else ((__half*)p)[i] = __float2half_rn(x);
}

template <int DT>
__global__ void __launch_bounds__(256) adamw_kernel(const __grid_constant__ AdamWLaunch L)
{
    pdl_enter();
    // the bias corrections of this step: every thread forms the same values
    const float b1t = __fmul_rn(L.bpow[0], L.b1), b2t = __fmul_rn(L.bpow[1], L.b2);
    const float decay = __fsub_rn(1.0f, __fmul_rn(L.lr, L.wd));
    const float c1 = __fsub_rn(1.0f, L.b1), c2 = __fsub_rn(1.0f, L.b2);
    const float step = __fdiv_rn(L.lr, __fsub_rn(1.0f, b1t));
    const float bc2s = __fsqrt_rn(__fsub_rn(1.0f, b2t));
    const long long total = L.start[L.count];
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        int lo = 0, hi = L.count - 1;  // the tensor holding element e
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (L.start[mid] <= e) lo = mid;
            else hi = mid - 1;
        }
        const long long i = e - L.start[lo];
        const float pi = ldp<DT>(L.p[lo], i), gi = ldp<DT>(L.g[lo], i);
        const float p1 = __fmul_rn(pi, decay);
        const float mi = __fadd_rn(__fmul_rn(L.b1, L.m[lo][i]), __fmul_rn(c1, gi));
        const float vi = __fadd_rn(__fmul_rn(L.b2, L.v[lo][i]), __fmul_rn(c2, __fmul_rn(gi, gi)));
        const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(vi), bc2s), L.eps);
        const float upd = __fdiv_rn(mi, denom);
        stp<DT>(L.p[lo], i, __fsub_rn(p1, __fmul_rn(step, upd)));
        L.m[lo][i] = mi;
        L.v[lo][i] = vi;
    }
}

__global__ void advance_powers(float* bpow, float b1, float b2)
{
    pdl_enter();
    bpow[0] = __fmul_rn(bpow[0], b1);
    bpow[1] = __fmul_rn(bpow[1], b2);
}

}  // namespace

}  // namespace psg

using namespace psg;

extern "C" psg_status psg_adamw_step(const psg_adamw_tensor* tensors, int n_tensors, int dtype, float lr, float beta1,
                                     float beta2, float eps, float weight_decay, float* d_beta_pow,
                                     int32_t* d_status, void* stream)
{
    (void)d_status;
    if (n_tensors < 0 || (n_tensors > 0 && (!tensors || !d_beta_pow))) return PSG_E_INVALID_ARG;
    if (dtype != PSG_F32 && dtype != PSG_BF16 && dtype != PSG_F16) return PSG_E_UNSUPPORTED_DTYPE;
    if (!(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f) || !(eps > 0.0f) || !(lr >= 0.0f))
        return PSG_E_INVALID_ARG;
    const int es = dtype_size(dtype);
    for (int k = 0; k < n_tensors; ++k) {
        const psg_adamw_tensor& t = tensors[k];
        if (t.numel < 0) return PSG_E_INVALID_ARG;
        if (t.numel > 0 && (!t.p || !t.g || !t.m || !t.v)) return PSG_E_INVALID_ARG;
        if ((uintptr_t)t.p % es || (uintptr_t)t.g % es || (uintptr_t)t.m % 4 || (uintptr_t)t.v % 4)
            return PSG_E_MISALIGNED;
    }
    if ((uintptr_t)d_beta_pow % 4) return PSG_E_MISALIGNED;
    cudaStream_t s = (cudaStream_t)stream;
    for (int g0 = 0; g0 < n_tensors; g0 += GROUP) {
        AdamWLaunch L;
        std::memset(&L, 0, sizeof(L));
        L.count = std::min(GROUP, n_tensors - g0);
        L.dtype = dtype;
        L.lr = lr;
        L.b1 = beta1;
        L.b2 = beta2;
        L.eps = eps;
        L.wd = weight_decay;
        L.bpow = d_beta_pow;
        for (int k = 0; k < L.count; ++k) {
            const psg_adamw_tensor& t = tensors[g0 + k];
            L.p[k] = t.p;
            L.g[k] = t.g;
            L.m[k] = t.m;
            L.v[k] = t.v;
            L.start[k + 1] = L.start[k] + t.numel;
        }
        const long long total = L.start[L.count];
        if (total == 0) continue;
        const int grid = (int)std::min<long long>((total + 255) / 256, (long long)num_sms() * 8);
        if (dtype == PSG_F32) launch(adamw_kernel<PSG_F32>, grid, 256, 0, s, L);
        else if (dtype == PSG_BF16) launch(adamw_kernel<PSG_BF16>, grid, 256, 0, s, L);
        else launch(adamw_kernel<PSG_F16>, grid, 256, 0, s, L);
    }
    launch(advance_powers, 1, 1, 0, s, d_beta_pow, beta1, beta2);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}
