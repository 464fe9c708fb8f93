// GATHER and SCATTER-add along dim 0 (sm_103a).
//
// GATHER (limn, "The op set"; the Embedding of "nn, optim and checkpoints"):
// one warp per output row copies src[idx[n], :] with 128-bit moves when both
// rows are contiguous and aligned.  An index outside [0, V) zero-fills its row
// and reports PSG_E_INDEX_OUT_OF_RANGE in the caller's status word.
//
// SCATTER-add, deterministic: limn's c device keeps a scatter's colliding adds
// serial ("Backends") and its cuda device uses atomics; here the colliding adds
// happen in ascending n without atomics.  The keys (idx[n] << 32 | n) are
// unique, so sorting them with a bitonic network gives one order no matter how
// the sort is scheduled; each run of equal idx is then added by one warp in
// that order into a float32 total seeded with the destination's value and
// rounded once (int32 wraps; float64 totals in double).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gather_scatter.h"
#include "launch_util.cuh"

namespace psg {

namespace {

constexpr int LOCAL_SORT = 2048;  // keys sorted per block in shared memory
constexpr unsigned long long BAD_HI = 0xffffffffull;

__device__ __forceinline__ void report(int32_t* st, int code)
{
    if (st) atomicCAS(st, 0, code);
}

// ---- GATHER ----------------------------------------------------------------
template <int ES>
__device__ __forceinline__ void copy_cell(char* d, const char* s)
{
    if constexpr (ES == 1) *(uint8_t*)d = *(const uint8_t*)s;
    else if constexpr (ES == 2) *(uint16_t*)d = *(const uint16_t*)s;
    else if constexpr (ES == 4) *(uint32_t*)d = *(const uint32_t*)s;
    else *(uint64_t*)d = *(const uint64_t*)s;
}
template <int ES>
__device__ __forceinline__ void zero_cell(char* d)
{
    if constexpr (ES == 1) *(uint8_t*)d = 0;
    else if constexpr (ES == 2) *(uint16_t*)d = 0;
    else if constexpr (ES == 4) *(uint32_t*)d = 0;
    else *(uint64_t*)d = 0;
}

template <int ES>
__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ GatherLaunch L)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * 8;
    for (int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); r < L.n; r += warps) {
        const int64_t v = L.idx[r];
        const bool ok = v >= 0 && v < L.V;
        if (!ok && lane == 0) report(L.status, PSG_E_INDEX_OUT_OF_RANGE);
        char* o = (char*)L.out + (L.out_offset + r * L.out_rs) * ES;
        const char* s = (const char*)L.src + (L.src_offset + (ok ? v : 0) * L.src_rs) * ES;
        if (L.vec16) {  // both rows contiguous and 16-byte aligned: D*ES is a multiple of 16
            const int64_t nv = L.D * ES / 16;
            for (int64_t i = lane; i < nv; i += 32)
                ((uint4*)o)[i] = ok ? __ldg((const uint4*)s + i) : make_uint4(0, 0, 0, 0);
        } else {
            for (int64_t i = lane; i < L.D; i += 32) {
                if (ok) copy_cell<ES>(o + i * L.out_cs * ES, s + i * L.src_cs * ES);
                else zero_cell<ES>(o + i * L.out_cs * ES);
            }
        }
    }
}

// ---- SCATTER: keys ---------------------------------------------------------
__global__ void make_keys(const int32_t* __restrict__ idx, int64_t n, int64_t V, int64_t npow2,
                          unsigned long long* __restrict__ keys, int32_t* status)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < npow2;
         i += (int64_t)gridDim.x * blockDim.x) {
        unsigned long long k;
        if (i < n) {
            const int64_t v = idx[i];
            if (v >= 0 && v < V) {
                k = ((unsigned long long)v << 32) | (unsigned long long)i;
            } else {
                k = (BAD_HI << 32) | (unsigned long long)i;  // sorts after every valid key
                report(status, PSG_E_INDEX_OUT_OF_RANGE);
            }
        } else {
            k = ~0ull;
        }
        keys[i] = k;
    }
}

__device__ __forceinline__ void cmp_swap(unsigned long long& a, unsigned long long& b, bool up)
{
    if ((a > b) == up) {
        const unsigned long long t = a;
        a = b;
        b = t;
    }
}

// all bitonic steps with j < LOCAL_SORT for stage k (k <= LOCAL_SORT: the
// whole local sort; k > LOCAL_SORT: the tail of a global merge stage)
__global__ void __launch_bounds__(1024) bitonic_local(unsigned long long* keys, int64_t npow2, int64_t kfrom)
{
    __shared__ unsigned long long s[LOCAL_SORT];
    const int64_t tile = (int64_t)blockIdx.x * LOCAL_SORT;
    const int t = threadIdx.x;
    const int m = npow2 < LOCAL_SORT ? (int)npow2 : LOCAL_SORT;
    for (int i = t; i < m; i += blockDim.x) s[i] = keys[tile + i];
    __syncthreads();
    const int64_t k0 = kfrom > 0 ? kfrom : 2;
    const int64_t k1 = kfrom > 0 ? kfrom : m;
    for (int64_t k = k0; k <= k1; k <<= 1) {
        for (int64_t j = (k < m ? k : m) >> 1; j > 0; j >>= 1) {
            for (int i = t; i < m / 2; i += blockDim.x) {
                // pair (a, a + j) with a having bit j clear
                const int a = (int)((i / j) * (2 * j) + (i % j));
                const int64_t ga = tile + a;
                const bool up = (ga & k) == 0;
                cmp_swap(s[a], s[a + j], up);
            }
            __syncthreads();
        }
    }
    for (int i = t; i < m; i += blockDim.x) keys[tile + i] = s[i];
}

// one global step (k, j) with j >= LOCAL_SORT: one thread per pair
__global__ void bitonic_global(unsigned long long* keys, int64_t npow2, int64_t k, int64_t j)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < npow2 / 2;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t a = (i / j) * (2 * j) + (i % j);
        const bool up = (a & k) == 0;
        unsigned long long x = keys[a], y = keys[a + j];
        if ((x > y) == up) {
            keys[a] = y;
            keys[a + j] = x;
        }
    }
}

// ---- SCATTER: segmented, ordered accumulation -------------------------------
template <typename T> struct Acc { typedef float A; };
template <> struct Acc<double> { typedef double A; };
template <> struct Acc<int32_t> { typedef int32_t A; };

template <int DT>
__device__ __forceinline__ float load_f(const void* p, int64_t o)
{
    if constexpr (DT == PSG_F32) return __ldg((const float*)p + o);
    else if constexpr (DT == PSG_BF16) return __uint_as_float(((uint32_t)__ldg((const uint16_t*)p + o)) << 16);
    else {
        const uint16_t h = __ldg((const uint16_t*)p + o);
        float r;
        asm("cvt.f32.f16 %0, %1;" : "=f"(r) : "h"(h));
        return r;
    }
}
template <int DT>
__device__ __forceinline__ void store_f(void* p, int64_t o, float v)
{
    if constexpr (DT == PSG_F32) ((float*)p)[o] = v;
    else if constexpr (DT == PSG_BF16) {
        uint16_t h;
        asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
        ((uint16_t*)p)[o] = h;
    } else {
        uint16_t h;
        asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(v));
        ((uint16_t*)p)[o] = h;
    }
}

template <int DT>
__global__ void __launch_bounds__(256) scatter_accumulate(const __grid_constant__ ScatterLaunch L,
                                                          const unsigned long long* __restrict__ keys)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * 8;
    for (int64_t p = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); p < L.n; p += warps) {
        const unsigned long long kp = keys[p];
        const unsigned long long hi = kp >> 32;
        if (hi == BAD_HI) continue;  // invalid index (or padding)
        if (p > 0 && (keys[p - 1] >> 32) == hi) continue;  // not the start of a run
        int64_t end = p + 1;
        while (end < L.n && (keys[end] >> 32) == hi) ++end;
        const int64_t v = (int64_t)hi;
        const int64_t drow = L.dst_offset + v * L.dst_rs;
        for (int64_t c = lane; c < L.D; c += 32) {
            const int64_t od = drow + c * L.dst_cs;
            if constexpr (DT == PSG_F64) {
                double acc = ((const double*)L.dst)[od];
                for (int64_t q = p; q < end; ++q) {
                    const int64_t n = (int64_t)(keys[q] & 0xffffffffull);
                    acc = __dadd_rn(acc, ((const double*)L.upd)[L.upd_offset + n * L.upd_rs + c * L.upd_cs]);
                }
                ((double*)L.dst)[od] = acc;
            } else if constexpr (DT == PSG_I32) {
                uint32_t acc = ((const uint32_t*)L.dst)[od];
                for (int64_t q = p; q < end; ++q) {
                    const int64_t n = (int64_t)(keys[q] & 0xffffffffull);
                    acc += ((const uint32_t*)L.upd)[L.upd_offset + n * L.upd_rs + c * L.upd_cs];
                }
                ((uint32_t*)L.dst)[od] = acc;
            } else {
                float acc = load_f<DT>(L.dst, od);
                for (int64_t q = p; q < end; ++q) {
                    const int64_t n = (int64_t)(keys[q] & 0xffffffffull);
                    acc = __fadd_rn(acc, load_f<DT>(L.upd, L.upd_offset + n * L.upd_rs + c * L.upd_cs));
                }
                store_f<DT>(L.dst, od, acc);
            }
        }
    }
}

int grid_for(const void* fn, int threads, int64_t work_blocks)
{
    const int per_sm = max_blocks_per_sm(fn, threads, 0);
    return (int)std::max<int64_t>(1, std::min<int64_t>(work_blocks, (int64_t)num_sms() * per_sm));
}

// Fixed scratch for psg_scatter_add_static: the sort keys of one call.  It is
// part of this library's device image, so every GPU that loads the library
// holds these 8 MiB until the process exits; the allocating scatter call never
// touches it.
__device__ __align__(256) unsigned long long g_static_keys[kStaticScatterKeys];

}  // namespace

// Device address of g_static_keys on the current device.  In host code the
// array's name only stands in for the symbol, so the address is asked from the
// runtime once per device (with that device current) and cached.
psg_status static_scatter_keys(unsigned long long** out)
{
    constexpr int MAX_DEV = 64;
    static std::mutex mu;
    static unsigned long long* ptrs[MAX_DEV];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return PSG_E_CUDA;
    std::lock_guard<std::mutex> g(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_keys) != cudaSuccess || !p) return PSG_E_CUDA;
        ptrs[dev] = (unsigned long long*)p;
    }
    *out = ptrs[dev];
    return PSG_OK;
}

int64_t scatter_npow2(int64_t n)
{
    int64_t p = 1;
    while (p < n) p <<= 1;
    return p;
}

psg_status launch_gather(const GatherLaunch& L, void* stream)
{
    if (L.n == 0) return PSG_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t blocks = (L.n + 7) / 8;
    switch (L.es) {
    case 1: gather_kernel<1><<<grid_for((const void*)gather_kernel<1>, 256, blocks), 256, 0, s>>>(L); break;
    case 2: gather_kernel<2><<<grid_for((const void*)gather_kernel<2>, 256, blocks), 256, 0, s>>>(L); break;
    case 4: gather_kernel<4><<<grid_for((const void*)gather_kernel<4>, 256, blocks), 256, 0, s>>>(L); break;
    default: gather_kernel<8><<<grid_for((const void*)gather_kernel<8>, 256, blocks), 256, 0, s>>>(L); break;
    }
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

psg_status launch_scatter(const ScatterLaunch& L, unsigned long long* keys, void* stream)
{
    if (L.n == 0) return PSG_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t np2 = scatter_npow2(L.n);
    make_keys<<<grid_for((const void*)make_keys, 256, (np2 + 255) / 256), 256, 0, s>>>(L.idx, L.n, L.V, np2,
                                                                                     keys, L.status);
    const int64_t tiles = (np2 + LOCAL_SORT - 1) / LOCAL_SORT;
    const int lthreads = 1024;
    bitonic_local<<<(unsigned)tiles, lthreads, 0, s>>>(keys, np2, 0);
    for (int64_t k = 2 * LOCAL_SORT; k <= np2; k <<= 1) {
        for (int64_t j = k >> 1; j >= LOCAL_SORT; j >>= 1)
            bitonic_global<<<grid_for((const void*)bitonic_global, 256, (np2 / 2 + 255) / 256), 256, 0, s>>>(
                keys, np2, k, j);
        bitonic_local<<<(unsigned)tiles, lthreads, 0, s>>>(keys, np2, k);
    }
    const int64_t blocks = (L.n + 7) / 8;
    switch (L.dtype) {
    case PSG_F32:
        scatter_accumulate<PSG_F32><<<grid_for((const void*)scatter_accumulate<PSG_F32>, 256, blocks), 256, 0, s>>>(L, keys);
        break;
    case PSG_BF16:
        scatter_accumulate<PSG_BF16><<<grid_for((const void*)scatter_accumulate<PSG_BF16>, 256, blocks), 256, 0, s>>>(L, keys);
        break;
    case PSG_F16:
        scatter_accumulate<PSG_F16><<<grid_for((const void*)scatter_accumulate<PSG_F16>, 256, blocks), 256, 0, s>>>(L, keys);
        break;
    case PSG_F64:
        scatter_accumulate<PSG_F64><<<grid_for((const void*)scatter_accumulate<PSG_F64>, 256, blocks), 256, 0, s>>>(L, keys);
        break;
    default:
        scatter_accumulate<PSG_I32><<<grid_for((const void*)scatter_accumulate<PSG_I32>, 256, blocks), 256, 0, s>>>(L, keys);
        break;
    }
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

}  // namespace psg
