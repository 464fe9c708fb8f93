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
// the sort is scheduled; each run of equal idx is then added in that order,
// one warp per (run, column segment), into a float32 total seeded with the
// destination's value and rounded once (int32 wraps; float64 totals in
// double).
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
            const int jj = (int)j;
            for (int i = t; i < m / 2; i += blockDim.x) {
                // pair (a, a + j) with a having bit j clear (j a power of two)
                const int a = ((i & ~(jj - 1)) << 1) | (i & (jj - 1));
                const int64_t ga = tile + a;
                const bool up = (ga & k) == 0;
                cmp_swap(s[a], s[a + j], up);
            }
            __syncthreads();
        }
    }
    for (int i = t; i < m; i += blockDim.x) keys[tile + i] = s[i];
}

// keys and the whole bitonic sort in one block for npow2 <= SMALL_SORT: the
// keys stay in shared memory for all log2(n) (log2(n) + 1) / 2 steps
constexpr int SMALL_SORT = 16384;
constexpr int SMALL_SORT_SMEM = SMALL_SORT * 8;  // 128 KB

template <int E>
__global__ void __launch_bounds__(1024) sort_small(const int32_t* __restrict__ idx, int64_t n, int64_t V, int npow2,
                                                   unsigned long long* __restrict__ keys, int32_t* status)
{
    // N = 1024 * E keys (padding ~0 sorts last); thread t holds keys
    // t*E .. t*E+E-1 in registers: a step (k, j) pairs i with i ^ j, inside the
    // thread for j < E, across lanes (shuffles) for j < 32 E, and through
    // shared memory above that
    extern __shared__ unsigned long long sk[];
    const int t = threadIdx.x;
    constexpr int N = 1024 * E;
    unsigned long long r[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int64_t i = (int64_t)t * E + e;
        unsigned long long k = ~0ull;
        if (i < n) {
            const int64_t v = idx[i];
            if (v >= 0 && v < V) {
                k = ((unsigned long long)v << 32) | (unsigned long long)i;
            } else {
                k = (BAD_HI << 32) | (unsigned long long)i;  // sorts after every valid key
                report(status, PSG_E_INDEX_OUT_OF_RANGE);
            }
        }
        r[e] = k;
    }
    for (int k = 2; k <= N; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= 32 * E) {
#pragma unroll
                for (int e = 0; e < E; ++e) sk[t * E + e] = r[e];
                __syncthreads();
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int i = t * E + e;
                    const unsigned long long q = sk[i ^ j];
                    const bool keep_min = ((i & j) == 0) == ((i & k) == 0);
                    r[e] = keep_min ? (q < r[e] ? q : r[e]) : (q > r[e] ? q : r[e]);
                }
                __syncthreads();
            } else if (j >= E) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int i = t * E + e;
                    const unsigned long long q = __shfl_xor_sync(0xffffffffu, r[e], j / E);
                    const bool keep_min = ((i & j) == 0) == ((i & k) == 0);
                    r[e] = keep_min ? (q < r[e] ? q : r[e]) : (q > r[e] ? q : r[e]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    if (e & j) continue;
                    const bool up = (((t * E + e) & k) == 0);
                    cmp_swap(r[e], r[e | j], up);
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e)
        if (t * E + e < npow2) keys[t * E + e] = r[e];
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
// SV<DT>: the running total's type A (float32 for the float widths, double
// for float64, uint32 for int32 so it wraps), loads of one cell or one
// 16-byte vector of cells as A, the add, and the store that rounds once.
template <int DT> struct SV;
template <> struct SV<PSG_F32> {
    typedef float A;
    static constexpr int ES = 4;
    static __device__ __forceinline__ A ld(const void* p, int64_t o) { return __ldg((const float*)p + o); }
    static __device__ __forceinline__ A add(A a, A b) { return __fadd_rn(a, b); }
    static __device__ __forceinline__ void st(void* p, int64_t o, A v) { ((float*)p)[o] = v; }
    static __device__ __forceinline__ void unpack(const uint4 u, A (&x)[16 / ES])
    {
        x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
        x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
    }
};
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
template <> struct SV<PSG_BF16> {
    typedef float A;
    static constexpr int ES = 2;
    static __device__ __forceinline__ A ld(const void* p, int64_t o)
    {
        return __uint_as_float(((uint32_t)__ldg((const uint16_t*)p + o)) << 16);
    }
    static __device__ __forceinline__ A add(A a, A b) { return __fadd_rn(a, b); }
    static __device__ __forceinline__ void st(void* p, int64_t o, A v)
    {
        uint16_t h;
        asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
        ((uint16_t*)p)[o] = h;
    }
    static __device__ __forceinline__ void unpack(const uint4 u, A (&x)[16 / ES])
    {
        x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
        x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
    }
};
__device__ __forceinline__ float f16_bits(uint16_t h)
{
    float r;
    asm("cvt.f32.f16 %0, %1;" : "=f"(r) : "h"(h));
    return r;
}
template <> struct SV<PSG_F16> {
    typedef float A;
    static constexpr int ES = 2;
    static __device__ __forceinline__ A ld(const void* p, int64_t o) { return f16_bits(__ldg((const uint16_t*)p + o)); }
    static __device__ __forceinline__ A add(A a, A b) { return __fadd_rn(a, b); }
    static __device__ __forceinline__ void st(void* p, int64_t o, A v)
    {
        uint16_t h;
        asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(v));
        ((uint16_t*)p)[o] = h;
    }
    static __device__ __forceinline__ void unpack(const uint4 u, A (&x)[16 / ES])
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = f16_bits((uint16_t)(w[i] & 0xffffu));
            x[2 * i + 1] = f16_bits((uint16_t)(w[i] >> 16));
        }
    }
};
template <> struct SV<PSG_F64> {
    typedef double A;
    static constexpr int ES = 8;
    static __device__ __forceinline__ A ld(const void* p, int64_t o) { return __ldg((const double*)p + o); }
    static __device__ __forceinline__ A add(A a, A b) { return __dadd_rn(a, b); }
    static __device__ __forceinline__ void st(void* p, int64_t o, A v) { ((double*)p)[o] = v; }
    static __device__ __forceinline__ void unpack(const uint4 u, A (&x)[16 / ES])
    {
        x[0] = __hiloint2double((int)u.y, (int)u.x);
        x[1] = __hiloint2double((int)u.w, (int)u.z);
    }
};
template <> struct SV<PSG_I32> {
    typedef uint32_t A;
    static constexpr int ES = 4;
    static __device__ __forceinline__ A ld(const void* p, int64_t o) { return __ldg((const uint32_t*)p + o); }
    static __device__ __forceinline__ A add(A a, A b) { return a + b; }
    static __device__ __forceinline__ void st(void* p, int64_t o, A v) { ((uint32_t*)p)[o] = v; }
    static __device__ __forceinline__ void unpack(const uint4 u, A (&x)[16 / ES])
    {
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    }
};

constexpr int SCATTER_UNROLL = 4;  // rows of a run loaded before they are added

// One warp per (run, column segment) item.  A segment is 32 * VPL columns,
// VPL cells per lane: a 16-byte vector when VEC (every update row contiguous
// and 16-byte aligned), else one cell.  The run's rows are added in
// ascending n into a total seeded with the destination's value; loading
// SCATTER_UNROLL rows ahead of the adds keeps more bytes in flight and
// leaves the order of the adds, hence the bits, unchanged.
template <int DT, bool VEC>
__global__ void __launch_bounds__(256) scatter_accumulate(const __grid_constant__ ScatterLaunch L,
                                                          const unsigned long long* __restrict__ keys,
                                                          int64_t nseg)
{
    typedef SV<DT> S;
    typedef typename S::A A;
    constexpr int VPL = VEC ? 16 / S::ES : 1;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * 8;
    const int64_t items = L.n * nseg;
    for (int64_t it = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); it < items; it += warps) {
        const int64_t p = it / nseg;
        const int64_t seg = it - p * nseg;
        const unsigned long long hi = keys[p] >> 32;
        if (hi == BAD_HI) continue;                          // invalid index (or padding)
        if (p > 0 && (keys[p - 1] >> 32) == hi) continue;    // not the start of a run
        // the run's end, 32 keys at a time (the item is the warp's: converged)
        int64_t end = p + 1;
        for (;;) {
            const int64_t q = end + lane;
            const unsigned same = __ballot_sync(0xffffffffu, q < L.n && (keys[q] >> 32) == hi);
            if (same != 0xffffffffu) {
                end += __ffs(~same) - 1;
                break;
            }
            end += 32;
        }
        const int64_t c0 = (seg * 32 + lane) * VPL;
        if (c0 >= L.D) continue;
        const int nv = L.D - c0 < VPL ? (int)(L.D - c0) : VPL;
        const int64_t drow = L.dst_offset + (int64_t)hi * L.dst_rs;
        A acc[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) acc[i] = i < nv ? S::ld(L.dst, drow + (c0 + i) * L.dst_cs) : A(0);
        for (int64_t q = p; q < end; q += SCATTER_UNROLL) {
            A x[SCATTER_UNROLL][VPL];
#pragma unroll
            for (int u = 0; u < SCATTER_UNROLL; ++u) {
                if (q + u >= end) break;
                const int64_t n = (int64_t)(keys[q + u] & 0xffffffffull);
                const int64_t o = L.upd_offset + n * L.upd_rs + c0 * L.upd_cs;
                if constexpr (VEC) {
                    if (nv == VPL) {
                        S::unpack(__ldg((const uint4*)((const char*)L.upd + o * S::ES)), x[u]);
                        continue;
                    }
                }
#pragma unroll
                for (int i = 0; i < VPL; ++i) x[u][i] = i < nv ? S::ld(L.upd, o + i * L.upd_cs) : A(0);
            }
#pragma unroll
            for (int u = 0; u < SCATTER_UNROLL; ++u) {
                if (q + u >= end) break;
#pragma unroll
                for (int i = 0; i < VPL; ++i) acc[i] = S::add(acc[i], x[u][i]);
            }
        }
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (i < nv) S::st(L.dst, drow + (c0 + i) * L.dst_cs, acc[i]);
    }
}

// Row-scan SCATTER-add for short update lists (n <= ROWSCAN_MAX_N): no sort.
// The block stages idx in shared memory; each warp owns one (destination
// row, column segment) item, lists the update rows n with idx[n] == row in
// ascending n (ballots over 32 indices at a time), then adds them in that
// order, ROWSCAN_AHEAD rows loaded ahead of the adds, into a total seeded
// with the destination's value and rounded once: the same adds in the same
// order as the sorted path, so the same bits.
constexpr int ROWSCAN_MAX_N = 16384;
constexpr int ROWSCAN_LIST = 256;    // listed rows per warp per round
constexpr int ROWSCAN_AHEAD = 8;

constexpr int ROWSCAN_WARPS = 4;

template <int DT, bool VEC>
__global__ void __launch_bounds__(ROWSCAN_WARPS * 32) scatter_rowscan(const __grid_constant__ ScatterLaunch L,
                                                                      int64_t nseg)
{
    typedef SV<DT> S;
    typedef typename S::A A;
    constexpr int VPL = VEC ? 16 / S::ES : 1;
    extern __shared__ int32_t sidx[];                      // [n] then [warps][ROWSCAN_LIST]
    int32_t* lists = sidx + ((L.n + 3) & ~3ll);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    bool bad = false;
#pragma unroll 8
    for (int64_t i = threadIdx.x; i < L.n; i += blockDim.x) {
        const int32_t v = __ldg(L.idx + i);
        const bool ok = v >= 0 && v < L.V;
        bad = bad || !ok;
        sidx[i] = ok ? v : -1;
    }
    if (bad && blockIdx.x == 0) report(L.status, PSG_E_INDEX_OUT_OF_RANGE);
    __syncthreads();
    int32_t* list = lists + w * ROWSCAN_LIST;
    const int64_t items = L.V * nseg;
    for (int64_t it = (int64_t)blockIdx.x * ROWSCAN_WARPS + w; it < items;
         it += (int64_t)gridDim.x * ROWSCAN_WARPS) {
        const int32_t row = (int32_t)(it / nseg);
        const int64_t seg = it - (int64_t)row * nseg;
        const int64_t c0 = (seg * 32 + lane) * VPL;
        const int nv = c0 >= L.D ? 0 : (L.D - c0 < VPL ? (int)(L.D - c0) : VPL);
        const int64_t drow = L.dst_offset + (int64_t)row * L.dst_rs;
        A acc[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) acc[i] = i < nv ? S::ld(L.dst, drow + (c0 + i) * L.dst_cs) : A(0);
        bool touched = false;
        int64_t base = 0;
        while (base < L.n) {
            // phase 1: the next (up to ROWSCAN_LIST) update rows aimed at `row`, ascending
            int cnt = 0;
            // four chunks of 32 indices per step: the shared loads go out together
            for (; base < L.n && cnt <= ROWSCAN_LIST - 128; base += 128) {
                int32_t v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t q = base + 32 * u + lane;
                    v[u] = q < L.n ? sidx[q] : -1;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const unsigned m = __ballot_sync(0xffffffffu, v[u] == row);
                    if (m) {
                        if (m & (1u << lane))
                            list[cnt + __popc(m & ((1u << lane) - 1u))] = (int32_t)(base + 32 * u + lane);
                        cnt += __popc(m);
                    }
                }
            }
            __syncwarp();
            // phase 2: add them in order, ROWSCAN_AHEAD rows in flight
            for (int e = 0; e < cnt; e += ROWSCAN_AHEAD) {
                A x[ROWSCAN_AHEAD][VPL];
#pragma unroll
                for (int u = 0; u < ROWSCAN_AHEAD; ++u) {
                    if (e + u >= cnt || nv == 0) break;
                    const int64_t o = L.upd_offset + (int64_t)list[e + u] * L.upd_rs + c0 * L.upd_cs;
                    if constexpr (VEC) {
                        if (nv == VPL) {
                            S::unpack(__ldg((const uint4*)((const char*)L.upd + o * S::ES)), x[u]);
                            continue;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < VPL; ++i) x[u][i] = i < nv ? S::ld(L.upd, o + i * L.upd_cs) : A(0);
                }
#pragma unroll
                for (int u = 0; u < ROWSCAN_AHEAD; ++u) {
                    if (e + u >= cnt || nv == 0) break;
#pragma unroll
                    for (int i = 0; i < VPL; ++i) acc[i] = S::add(acc[i], x[u][i]);
                }
            }
            touched = touched || cnt > 0;
            __syncwarp();
        }
        // rows nothing lands on keep their bits (no write at all)
        if (touched) {
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (i < nv) S::st(L.dst, drow + (c0 + i) * L.dst_cs, acc[i]);
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

template <int DT>
static void launch_accumulate(const ScatterLaunch& L, const unsigned long long* keys, cudaStream_t s)
{
    constexpr int ES = SV<DT>::ES;
    const bool vec = L.upd_cs == 1 && ((uintptr_t)L.upd + (uint64_t)L.upd_offset * ES) % 16 == 0 &&
                     ((uint64_t)L.upd_rs * ES) % 16 == 0;
    const int64_t seg_cols = 32 * (vec ? 16 / ES : 1);
    const int64_t nseg = (L.D + seg_cols - 1) / seg_cols;
    const int64_t blocks = (L.n * nseg + 7) / 8;
    if (nseg == 0) return;
    if (vec)
        scatter_accumulate<DT, true><<<grid_for((const void*)scatter_accumulate<DT, true>, 256, blocks), 256, 0, s>>>(
            L, keys, nseg);
    else
        scatter_accumulate<DT, false><<<grid_for((const void*)scatter_accumulate<DT, false>, 256, blocks), 256, 0,
                                        s>>>(L, keys, nseg);
}

template <int DT>
static psg_status launch_rowscan(const ScatterLaunch& L, cudaStream_t s)
{
    constexpr int ES = SV<DT>::ES;
    const bool vec = L.upd_cs == 1 && ((uintptr_t)L.upd + (uint64_t)L.upd_offset * ES) % 16 == 0 &&
                     ((uint64_t)L.upd_rs * ES) % 16 == 0;
    const int64_t seg_cols = 32 * (vec ? 16 / ES : 1);
    const int64_t nseg = (L.D + seg_cols - 1) / seg_cols;
    if (nseg == 0) return PSG_OK;
    const size_t smem = (size_t)(((L.n + 3) & ~3ll) + ROWSCAN_WARPS * ROWSCAN_LIST) * 4;
    const int64_t blocks =
        std::min<int64_t>((L.V * nseg + ROWSCAN_WARPS - 1) / ROWSCAN_WARPS, (int64_t)num_sms() * 4);
    static std::once_flag once[2];
    static cudaError_t err[2] = {cudaSuccess, cudaSuccess};
    const void* fn = vec ? (const void*)scatter_rowscan<DT, true> : (const void*)scatter_rowscan<DT, false>;
    std::call_once(once[vec ? 1 : 0], [fn] {
        err[fn == (const void*)scatter_rowscan<DT, true> ? 1 : 0] =
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    });
    if (err[vec ? 1 : 0] != cudaSuccess) return PSG_E_CUDA;
    if (vec) scatter_rowscan<DT, true><<<(unsigned)blocks, ROWSCAN_WARPS * 32, smem, s>>>(L, nseg);
    else scatter_rowscan<DT, false><<<(unsigned)blocks, ROWSCAN_WARPS * 32, smem, s>>>(L, nseg);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

// the row scan reads all n indices once per (row, segment) item from shared
// memory: worth it while V * n stays small against one sort of n keys
static bool use_rowscan(const ScatterLaunch& L)
{
    return L.n <= ROWSCAN_MAX_N && L.V <= 4096 && L.V * L.n <= (int64_t)1 << 24;
}

psg_status launch_scatter(const ScatterLaunch& L, unsigned long long* keys, void* stream)
{
    if (L.n == 0) return PSG_OK;
    cudaStream_t s = (cudaStream_t)stream;
    if (use_rowscan(L)) {
        switch (L.dtype) {
        case PSG_F32: return launch_rowscan<PSG_F32>(L, s);
        case PSG_BF16: return launch_rowscan<PSG_BF16>(L, s);
        case PSG_F16: return launch_rowscan<PSG_F16>(L, s);
        case PSG_F64: return launch_rowscan<PSG_F64>(L, s);
        default: return launch_rowscan<PSG_I32>(L, s);
        }
    }
    const int64_t np2 = scatter_npow2(L.n);
    if (np2 <= SMALL_SORT) {
        static std::once_flag once;
        static cudaError_t err = cudaSuccess;
        std::call_once(once, [] {
            const void* fns[5] = {(const void*)sort_small<1>, (const void*)sort_small<2>, (const void*)sort_small<4>,
                                  (const void*)sort_small<8>, (const void*)sort_small<16>};
            for (const void* f : fns)
                if (err == cudaSuccess)
                    err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SMALL_SORT_SMEM);
        });
        if (err != cudaSuccess) return PSG_E_CUDA;
        const int N = np2 < 1024 ? 1024 : (int)np2;
        const size_t sm = (size_t)N * 8;
        switch (N / 1024) {
        case 1: sort_small<1><<<1, 1024, sm, s>>>(L.idx, L.n, L.V, (int)np2, keys, L.status); break;
        case 2: sort_small<2><<<1, 1024, sm, s>>>(L.idx, L.n, L.V, (int)np2, keys, L.status); break;
        case 4: sort_small<4><<<1, 1024, sm, s>>>(L.idx, L.n, L.V, (int)np2, keys, L.status); break;
        case 8: sort_small<8><<<1, 1024, sm, s>>>(L.idx, L.n, L.V, (int)np2, keys, L.status); break;
        default: sort_small<16><<<1, 1024, sm, s>>>(L.idx, L.n, L.V, (int)np2, keys, L.status); break;
        }
    } else {
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
    }
    switch (L.dtype) {
    case PSG_F32: launch_accumulate<PSG_F32>(L, keys, s); break;
    case PSG_BF16: launch_accumulate<PSG_BF16>(L, keys, s); break;
    case PSG_F16: launch_accumulate<PSG_F16>(L, keys, s); break;
    case PSG_F64: launch_accumulate<PSG_F64>(L, keys, s); break;
    default: launch_accumulate<PSG_I32>(L, keys, s); break;
    }
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

}  // namespace psg
