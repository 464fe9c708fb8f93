// GATHER and SCATTER-add along dim 0 (sm_103a).
//
// GATHER (limn, "The op set"; the Embedding of "nn, optim and checkpoints"):
// one warp per output row copies src[idx[n], :] with 128-bit moves when both
// rows are contiguous and aligned.  An index outside [0, V) zero-fills its row
// and reports PSG_E_INDEX_OUT_OF_RANGE in the caller's status word.
//
// SCATTER-add, deterministic: limn's c device keeps a scatter's colliding adds
// serial ("Backends") and its cuda device uses atomics; here the colliding adds
// happen in ascending n without atomics.  The update rows are ordered by
// destination with a stable sort (one block's radix sort in shared memory for
// lists up to kScatterPlanMaxN; 64-bit keys idx << 32 | n through a bitonic
// network above that), so equal destinations keep ascending n whatever the
// schedule; each run of equal destination is then added in that order, one
// warp per (run, column segment), into a float32 total seeded with the
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
    pdl_enter();
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
    pdl_enter();
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
    pdl_enter();
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

// one global step (k, j) with j >= LOCAL_SORT: one thread per pair
__global__ void bitonic_global(unsigned long long* keys, int64_t npow2, int64_t k, int64_t j)
{
    pdl_enter();
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

// the narrow ints keep a wrapping 32-bit total too and store its low bits
// (addition modulo 2^width gives the same bits in any grouping)
template <> struct SV<PSG_I16> {
    typedef uint32_t A;
    static constexpr int ES = 2;
    static __device__ __forceinline__ A ld(const void* p, int64_t o) { return (uint32_t)(int32_t)__ldg((const int16_t*)p + o); }
    static __device__ __forceinline__ A add(A a, A b) { return a + b; }
    static __device__ __forceinline__ void st(void* p, int64_t o, A v) { ((uint16_t*)p)[o] = (uint16_t)(v & 0xffffu); }
    static __device__ __forceinline__ void unpack(const uint4 u, A (&x)[16 / ES])
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = (uint32_t)(int32_t)(int16_t)(w[i] & 0xffffu);
            x[2 * i + 1] = (uint32_t)(int32_t)(int16_t)(w[i] >> 16);
        }
    }
};
template <> struct SV<PSG_I8> {
    typedef uint32_t A;
    static constexpr int ES = 1;
    static __device__ __forceinline__ A ld(const void* p, int64_t o) { return (uint32_t)(int32_t)__ldg((const int8_t*)p + o); }
    static __device__ __forceinline__ A add(A a, A b) { return a + b; }
    static __device__ __forceinline__ void st(void* p, int64_t o, A v) { ((uint8_t*)p)[o] = (uint8_t)(v & 0xffu); }
    static __device__ __forceinline__ void unpack(const uint4 u, A (&x)[16 / ES])
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (uint32_t)(int32_t)(int8_t)((w[i >> 2] >> (8 * (i & 3))) & 0xffu);
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
    pdl_enter();
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

// ---- SCATTER, n <= kScatterPlanMaxN: one block plans the order --------------
// One block loads the indices and orders the update rows by destination with
// a stable LSD radix sort in shared memory (4-bit digits over only the bits
// the largest key needs; indices already in order skip it).  Stability keeps
// ascending n inside each destination, so the order is the one the serial
// loop adds in.  The block writes the permutation and the runs of equal
// destination; scatter_runs then adds each run in that order.
constexpr int PLAN_THREADS = 512;
constexpr int PLAN_SMEM = kScatterPlanMaxN * 4 + 2 * kScatterPlanMaxN * 2;  // keys + two uint16 orders

struct PlanOut {
    int32_t* hdr;        // [0]: number of runs
    int32_t* perm;       // [n]: update rows in (destination, n) order
    int32_t* run_v;      // [n]: destination row of run r
    int32_t* run_start;  // [n + 1]: run r is perm[run_start[r] .. run_start[r + 1])
};

PlanOut plan_layout(void* ws, int64_t n)
{
    int32_t* b = (int32_t*)ws;
    return PlanOut{b, b + 4, b + 4 + n, b + 4 + 2 * n};
}

__device__ __forceinline__ unsigned long long warp_incl_scan(unsigned long long x, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// x: this thread's counts (NW packed words) -> their exclusive prefix over
// the threads before it; tot: the block's totals.  sh: [33 * NW] words.
template <int NW>
__device__ __forceinline__ void block_scan(unsigned long long (&x)[NW], unsigned long long (&tot)[NW],
                                           unsigned long long* sh)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    unsigned long long inc[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) inc[k] = warp_incl_scan(x[k], lane);
    if (lane == 31) {
#pragma unroll
        for (int k = 0; k < NW; ++k) sh[w * NW + k] = inc[k];
    }
    __syncthreads();
    if (w == 0) {
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const unsigned long long v = lane < (PLAN_THREADS >> 5) ? sh[lane * NW + k] : 0ull;
            const unsigned long long vi = warp_incl_scan(v, lane);
            if (lane < (PLAN_THREADS >> 5)) sh[lane * NW + k] = vi - v;
            if (lane == 31) sh[32 * NW + k] = vi;
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < NW; ++k) {
        tot[k] = sh[32 * NW + k];
        x[k] = sh[w * NW + k] + inc[k] - x[k];
    }
    __syncthreads();
}

// 16 bins as four words of four 16-bit counts (a bin never holds more than
// kScatterPlanMaxN = 2^14 rows, so no count carries into its neighbour)
__device__ __forceinline__ void bin_add(unsigned long long (&c)[4], int d)
{
    const unsigned long long inc = 1ull << (16 * (d & 3));
#pragma unroll
    for (int k = 0; k < 4; ++k) c[k] += (d >> 2) == k ? inc : 0ull;
}
__device__ __forceinline__ int bin_get(const unsigned long long (&c)[4], int d)
{
    const int k = d >> 2;
    const unsigned long long w = k == 0 ? c[0] : k == 1 ? c[1] : k == 2 ? c[2] : c[3];
    return (int)((w >> (16 * (d & 3))) & 0xffffull);
}

constexpr int PLAN_E = kScatterPlanMaxN / PLAN_THREADS;  // positions a thread owns, at most

__global__ void __launch_bounds__(PLAN_THREADS) scatter_plan(const int32_t* __restrict__ idx, int n, int64_t V,
                                                             PlanOut P, int32_t* status)
{
    pdl_enter();
    extern __shared__ uint32_t key[];                        // [kScatterPlanMaxN]
    uint16_t* ord0 = (uint16_t*)(key + kScatterPlanMaxN);   // [kScatterPlanMaxN] x 2
    uint16_t* ord1 = ord0 + kScatterPlanMaxN;
    __shared__ unsigned long long sh[33 * 4];
    __shared__ int base[16];
    const int t = threadIdx.x;
    // this thread's positions: a contiguous slice, so a thread-ordered prefix is position order
    const int E = (n + PLAN_THREADS - 1) / PLAN_THREADS;
    const int p0 = min(n, t * E), cnt = min(n, p0 + E) - p0;
    // key of update row i: its destination, or V (after every valid one) if out of range;
    // the slice's loads all go out before the first is used
    uint32_t kv[PLAN_E];
#pragma unroll
    for (int e = 0; e < PLAN_E; ++e)
        if (e < cnt) kv[e] = (uint32_t)__ldg(idx + p0 + e);
    bool bad = false, unsorted = false;
#pragma unroll
    for (int e = 0; e < PLAN_E; ++e) {
        if (e < cnt) {
            const int32_t v = (int32_t)kv[e];
            const bool ok = v >= 0 && (int64_t)v < V;
            bad = bad || !ok;
            kv[e] = ok ? (uint32_t)v : (uint32_t)V;
            key[p0 + e] = kv[e];
            ord0[p0 + e] = (uint16_t)(p0 + e);
            if (e > 0) unsorted = unsorted || kv[e] < kv[e - 1];
        }
    }
    const bool any_bad = __syncthreads_or(bad);
    if (bad) report(status, PSG_E_INDEX_OUT_OF_RANGE);
    if (cnt > 0 && p0 > 0) unsorted = unsorted || kv[0] < key[p0 - 1];
    if (!__syncthreads_or(unsorted)) {
        // already in order (the structured case): the run kernels walk idx itself
        if (t == 0) P.hdr[0] = -1;
        return;
    }
    const uint32_t kmax = any_bad ? (uint32_t)V : (uint32_t)(V - 1);
    const int bits = kmax ? 32 - __clz(kmax) : 0;
    uint16_t* src = ord0;
    uint16_t* dst = ord1;
    for (int shift = 0; shift < bits; shift += 4) {
        // w[e]: row (low 16 bits) and its digit (bits 16..19)
        uint32_t w[PLAN_E];
#pragma unroll
        for (int e = 0; e < PLAN_E; ++e)
            if (e < cnt) w[e] = src[p0 + e];
#pragma unroll
        for (int e = 0; e < PLAN_E; ++e)
            if (e < cnt) w[e] |= ((key[w[e]] >> shift) & 15u) << 16;
        unsigned long long c[4] = {0ull, 0ull, 0ull, 0ull}, tot[4];
#pragma unroll
        for (int e = 0; e < PLAN_E; ++e)
            if (e < cnt) bin_add(c, (int)(w[e] >> 16));
        block_scan<4>(c, tot, sh);
        if (t < 16) {
            int b = 0;
#pragma unroll
            for (int d = 0; d < 16; ++d) b += d < t ? bin_get(tot, d) : 0;
            base[t] = b;
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < PLAN_E; ++e) {
            if (e < cnt) {
                const int d = (int)(w[e] >> 16);
                dst[base[d] + bin_get(c, d)] = (uint16_t)(w[e] & 0xffffu);
                bin_add(c, d);
            }
        }
        __syncthreads();
        uint16_t* x = src;
        src = dst;
        dst = x;
    }
    // runs: a valid row whose key differs from the previous position's
    uint32_t row[PLAN_E];
#pragma unroll
    for (int e = 0; e < PLAN_E; ++e)
        if (e < cnt) row[e] = src[p0 + e];
#pragma unroll
    for (int e = 0; e < PLAN_E; ++e)
        if (e < cnt) kv[e] = key[row[e]];
    uint32_t prev = (cnt > 0 && p0 > 0) ? key[src[p0 - 1]] : 0xffffffffu;
    unsigned long long rc[2] = {0ull, 0ull}, rt[2];
    unsigned starts = 0;  // bit e: position p0 + e starts a run (PLAN_E <= 32)
#pragma unroll
    for (int e = 0; e < PLAN_E; ++e) {
        if (e < cnt) {
            const uint32_t pk = e == 0 ? prev : kv[e - 1];
            if ((int64_t)kv[e] < V) {
                rc[1] += 1;
                if (p0 + e == 0 || pk != kv[e]) {
                    rc[0] += 1;
                    starts |= 1u << e;
                }
            }
        }
    }
    block_scan<2>(rc, rt, sh);
    int r = (int)rc[0];
#pragma unroll
    for (int e = 0; e < PLAN_E; ++e) {
        if (e < cnt) {
            P.perm[p0 + e] = (int32_t)row[e];
            if (starts & (1u << e)) {
                P.run_v[r] = (int32_t)kv[e];
                P.run_start[r] = p0 + e;
                ++r;
            }
        }
    }
    if (t == 0) {
        P.hdr[0] = (int32_t)rt[0];
        P.run_start[rt[0]] = (int32_t)rt[1];  // the valid rows end the last run
    }
}

constexpr int RUN_AHEAD = 16;  // update rows of a run loaded before they are added

// One warp per (run, column segment), as scatter_accumulate, over the planned runs.
template <int DT, bool VEC>
__global__ void __launch_bounds__(256) scatter_runs(const __grid_constant__ ScatterLaunch L, const PlanOut P,
                                                    int64_t nseg)
{
    pdl_enter();
    typedef SV<DT> S;
    typedef typename S::A A;
    constexpr int VPL = VEC ? 16 / S::ES : 1;
    const int lane = threadIdx.x & 31;
    const int R = P.hdr[0];
    const bool walk = R < 0;  // indices already in order: the runs are idx's own stretches
    const int64_t items = (walk ? L.n : (int64_t)R) * nseg;
    for (int64_t it = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); it < items; it += (int64_t)gridDim.x * 8) {
        const int64_t r = it / nseg;
        const int64_t seg = it - r * nseg;
        int q0, q1;
        int64_t v;
        if (walk) {
            // the item is the whole warp's: these exits and the ballots are uniform
            v = __ldg(L.idx + r);
            if (v < 0 || v >= L.V || (r > 0 && __ldg(L.idx + r - 1) == v)) continue;
            q0 = (int)r;
            q1 = q0 + 1;
            for (;;) {
                const int64_t q = q1 + lane;
                const unsigned same = __ballot_sync(0xffffffffu, q < L.n && __ldg(L.idx + q) == v);
                if (same != 0xffffffffu) {
                    q1 += __ffs(~same) - 1;
                    break;
                }
                q1 += 32;
            }
        } else {
            q0 = P.run_start[r];
            q1 = P.run_start[r + 1];
            v = P.run_v[r];
        }
        const int64_t c0 = (seg * 32 + lane) * VPL;
        // lanes past the row's end stay in the loop (the shuffles below need the whole warp)
        const int nv = c0 >= L.D ? 0 : (L.D - c0 < VPL ? (int)(L.D - c0) : VPL);
        const int64_t drow = L.dst_offset + v * L.dst_rs;
        A acc[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) acc[i] = i < nv ? S::ld(L.dst, drow + (c0 + i) * L.dst_cs) : A(0);
        for (int q = q0; q < q1; q += 32) {
            // 32 update rows of the run: one coalesced load of their numbers, shared by shuffles
            const int m = min(32, q1 - q);
            const int my = lane < m ? (walk ? q + lane : __ldg(P.perm + q + lane)) : 0;
            for (int h = 0; h < m; h += RUN_AHEAD) {
                int rows[RUN_AHEAD];
#pragma unroll
                for (int u = 0; u < RUN_AHEAD; ++u) rows[u] = __shfl_sync(0xffffffffu, my, (h + u) & 31);
                // one cell at a time (a lane's cell, or the ragged last vector segment)
                auto cells = [&]() {
#pragma unroll
                    for (int i = 0; i < VPL; ++i) {
                        if (i >= nv) break;
                        A x[RUN_AHEAD];
#pragma unroll
                        for (int u = 0; u < RUN_AHEAD; ++u)
                            if (h + u < m)
                                x[u] = S::ld(L.upd, L.upd_offset + (int64_t)rows[u] * L.upd_rs + (c0 + i) * L.upd_cs);
#pragma unroll
                        for (int u = 0; u < RUN_AHEAD; ++u)
                            if (h + u < m) acc[i] = S::add(acc[i], x[u]);
                    }
                };
                if constexpr (VEC) {
                    if (nv == VPL) {
                        uint4 raw[RUN_AHEAD];
#pragma unroll
                        for (int u = 0; u < RUN_AHEAD; ++u)
                            if (h + u < m)
                                raw[u] = __ldg((const uint4*)((const char*)L.upd +
                                                              (L.upd_offset + (int64_t)rows[u] * L.upd_rs + c0) * S::ES));
#pragma unroll
                        for (int u = 0; u < RUN_AHEAD; ++u) {
                            if (h + u < m) {
                                A x[VPL];
                                S::unpack(raw[u], x);
#pragma unroll
                                for (int i = 0; i < VPL; ++i) acc[i] = S::add(acc[i], x[i]);
                            }
                        }
                    } else {
                        cells();
                    }
                } else {
                    cells();
                }
            }
        }
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (i < nv) S::st(L.dst, drow + (c0 + i) * L.dst_cs, acc[i]);
    }
}

// ---- SCATTER onto few destination rows: one block owns a row ----------------
// While V * n stays small, block (row, column chunk) scans all n indices for
// its row (16-byte loads; L2 serves the repeats), lists the matching update
// rows in ascending n in shared memory, and adds them in that order: no sort,
// no workspace, the same adds as the serial loop.
constexpr int OWNER_THREADS = 256;
constexpr int64_t OWNER_MAX_V = 4096;
constexpr int64_t OWNER_MAX_VN = int64_t(1) << 24;

constexpr int OWNER_R = (int)(kScatterPlanMaxN / (OWNER_THREADS * 4));  // 16-byte index loads a thread makes
constexpr int OWNER_AHEAD = 32;  // listed rows loaded before they are added

// two 16-bit cells of a 4-byte word as the running-total type
template <int DT>
__device__ __forceinline__ void unpack_pair(uint32_t u, float (&x)[2])
{
    if constexpr (DT == PSG_BF16) {
        x[0] = __uint_as_float(u << 16);
        x[1] = __uint_as_float(u & 0xffff0000u);
    } else {
        x[0] = f16_bits((uint16_t)(u & 0xffffu));
        x[1] = f16_bits((uint16_t)(u >> 16));
    }
}

// PAIR: 16-bit cells, two a thread through one 4-byte load (rows contiguous
// and 4-byte aligned); otherwise one cell a thread
template <int DT, bool PAIR>
__global__ void __launch_bounds__(OWNER_THREADS) scatter_owner(const __grid_constant__ ScatterLaunch L, int64_t ncb,
                                                               int idx16)
{
    pdl_enter();
    typedef SV<DT> S;
    typedef typename S::A A;
    constexpr int VPL = PAIR ? 2 : 1;
    extern __shared__ int32_t list[];  // [n]: update rows aimed at this row, ascending
    __shared__ int wsum[OWNER_THREADS / 32];
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int64_t row = blockIdx.x / ncb, cb = blockIdx.x - row * ncb;
    // 1. list: thread t owns the contiguous indices e0 .. e0 + 4R - 1, loaded all at once
    const int R = (int)((L.n + OWNER_THREADS * 4 - 1) / (OWNER_THREADS * 4));
    const int64_t e0 = (int64_t)t * 4 * R;
    int4 q[OWNER_R];
#pragma unroll
    for (int r = 0; r < OWNER_R; ++r) {
        if (r < R) {
            const int64_t i0 = e0 + 4 * r;
            if (idx16 && i0 + 3 < L.n) {
                q[r] = __ldg((const int4*)(L.idx + i0));
            } else {
                q[r].x = i0 < L.n ? __ldg(L.idx + i0) : 0;
                q[r].y = i0 + 1 < L.n ? __ldg(L.idx + i0 + 1) : 0;
                q[r].z = i0 + 2 < L.n ? __ldg(L.idx + i0 + 2) : 0;
                q[r].w = i0 + 3 < L.n ? __ldg(L.idx + i0 + 3) : 0;
            }
        }
    }
    unsigned long long hit = 0;  // bit k: index e0 + k is aimed at this row
    bool bad = false;
#pragma unroll
    for (int r = 0; r < OWNER_R; ++r) {
        if (r < R) {
            const int32_t v[4] = {q[r].x, q[r].y, q[r].z, q[r].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (e0 + 4 * r + j < L.n) {
                    bad = bad || v[j] < 0 || (int64_t)v[j] >= L.V;
                    if ((int64_t)v[j] == row) hit |= 1ull << (4 * r + j);
                }
            }
        }
    }
    if (bad && blockIdx.x == 0) report(L.status, PSG_E_INDEX_OUT_OF_RANGE);  // block 0 saw every index
    const int c = __popcll(hit);
    int x = c;  // inclusive prefix over the warp, then over the warps before
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    int off = x - c, total = 0;
#pragma unroll
    for (int k = 0; k < OWNER_THREADS / 32; ++k) {
        const int sk = wsum[k];
        off += k < w ? sk : 0;
        total += sk;
    }
    while (hit) {
        list[off++] = (int32_t)(e0 + __ffsll((long long)hit) - 1);
        hit &= hit - 1;
    }
    __syncthreads();
    if (total == 0) return;  // a row nothing lands on keeps its bits (no write)
    // 2. add them in order; thread t owns VPL cells of the chunk
    const int64_t c0 = (cb * OWNER_THREADS + t) * VPL;
    if (c0 >= L.D) return;
    const int nv = L.D - c0 < VPL ? (int)(L.D - c0) : VPL;
    const int64_t drow = L.dst_offset + row * L.dst_rs;
    A acc[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) acc[i] = i < nv ? S::ld(L.dst, drow + (c0 + i) * L.dst_cs) : A(0);
    for (int q0 = 0; q0 < total; q0 += OWNER_AHEAD) {
        if (PAIR && nv == 2) {
            uint32_t raw[OWNER_AHEAD];
#pragma unroll
            for (int u = 0; u < OWNER_AHEAD; ++u)
                if (q0 + u < total)
                    raw[u] = __ldg((const uint32_t*)((const char*)L.upd +
                                                     (L.upd_offset + (int64_t)list[q0 + u] * L.upd_rs + c0) * S::ES));
#pragma unroll
            for (int u = 0; u < OWNER_AHEAD; ++u) {
                if (q0 + u < total) {
                    float xx[2];
                    unpack_pair<DT>(raw[u], xx);
                    acc[0] = S::add(acc[0], xx[0]);
                    acc[VPL - 1] = S::add(acc[VPL - 1], xx[1]);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                if (i >= nv) break;
                A xx[OWNER_AHEAD];
#pragma unroll
                for (int u = 0; u < OWNER_AHEAD; ++u)
                    if (q0 + u < total)
                        xx[u] = S::ld(L.upd, L.upd_offset + (int64_t)list[q0 + u] * L.upd_rs + (c0 + i) * L.upd_cs);
#pragma unroll
                for (int u = 0; u < OWNER_AHEAD; ++u)
                    if (q0 + u < total) acc[i] = S::add(acc[i], xx[u]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (i < nv) S::st(L.dst, drow + (c0 + i) * L.dst_cs, acc[i]);
}

// Rows of a few cells (D <= NARROW_D): one thread per run, every cell of the row.
constexpr int NARROW_D = 4;

template <int DT>
__global__ void __launch_bounds__(256) scatter_runs_narrow(const __grid_constant__ ScatterLaunch L, const PlanOut P)
{
    pdl_enter();
    typedef SV<DT> S;
    typedef typename S::A A;
    const int R = P.hdr[0];
    const bool walk = R < 0;  // indices already in order: the runs are idx's own stretches
    const int64_t items = walk ? L.n : (int64_t)R;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < items; r += (int64_t)gridDim.x * blockDim.x) {
        int q0, q1;
        int64_t v;
        if (walk) {
            v = __ldg(L.idx + r);
            if (v < 0 || v >= L.V || (r > 0 && __ldg(L.idx + r - 1) == v)) continue;
            q0 = (int)r;
            q1 = q0 + 1;
            while (q1 < L.n && __ldg(L.idx + q1) == v) ++q1;
        } else {
            q0 = P.run_start[r];
            q1 = P.run_start[r + 1];
            v = P.run_v[r];
        }
        const int64_t drow = L.dst_offset + v * L.dst_rs;
        A acc[NARROW_D];
#pragma unroll
        for (int i = 0; i < NARROW_D; ++i) acc[i] = i < L.D ? S::ld(L.dst, drow + i * L.dst_cs) : A(0);
        for (int q = q0; q < q1; ++q) {
            const int64_t o = L.upd_offset + (int64_t)(walk ? q : __ldg(P.perm + q)) * L.upd_rs;
#pragma unroll
            for (int i = 0; i < NARROW_D; ++i)
                if (i < L.D) acc[i] = S::add(acc[i], S::ld(L.upd, o + i * L.upd_cs));
        }
#pragma unroll
        for (int i = 0; i < NARROW_D; ++i)
            if (i < L.D) S::st(L.dst, drow + i * L.dst_cs, acc[i]);
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

size_t scatter_workspace_bytes(int64_t n)
{
    if (n <= 0) return 0;
    if (n <= kScatterPlanMaxN) return (size_t)(4 + 3 * n + 1) * 4;  // plan_layout
    return (size_t)scatter_npow2(n) * sizeof(unsigned long long);
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
    case 1: launch(gather_kernel<1>, grid_for((const void*)gather_kernel<1>, 256, blocks), 256, 0, s, L); break;
    case 2: launch(gather_kernel<2>, grid_for((const void*)gather_kernel<2>, 256, blocks), 256, 0, s, L); break;
    case 4: launch(gather_kernel<4>, grid_for((const void*)gather_kernel<4>, 256, blocks), 256, 0, s, L); break;
    default: launch(gather_kernel<8>, grid_for((const void*)gather_kernel<8>, 256, blocks), 256, 0, s, L); break;
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
        launch(scatter_accumulate<DT, true>, grid_for((const void*)scatter_accumulate<DT, true>, 256, blocks), 256, 0, s, L, keys, nseg);
    else
        launch(scatter_accumulate<DT, false>, grid_for((const void*)scatter_accumulate<DT, false>, 256, blocks), 256, 0, s, L, keys, nseg);
}

template <int DT>
static psg_status launch_planned(const ScatterLaunch& L, void* ws, cudaStream_t s)
{
    if (set_max_dynamic_smem((const void*)scatter_plan, PLAN_SMEM) != cudaSuccess) return PSG_E_CUDA;
    const PlanOut P = plan_layout(ws, L.n);
    launch(scatter_plan, 1, PLAN_THREADS, PLAN_SMEM, s, L.idx, (int)L.n, L.V, P, L.status);
    const int64_t runs = std::min<int64_t>(L.n, L.V);  // at most this many runs
    if (L.D <= NARROW_D) {
        launch(scatter_runs_narrow<DT>, grid_for((const void*)scatter_runs_narrow<DT>, 256, (runs + 255) / 256), 256, 0, s, L, P);
        return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
    }
    constexpr int ES = SV<DT>::ES;
    const bool vec = L.upd_cs == 1 && ((uintptr_t)L.upd + (uint64_t)L.upd_offset * ES) % 16 == 0 &&
                     ((uint64_t)L.upd_rs * ES) % 16 == 0;
    const int64_t seg_cols = 32 * (vec ? 16 / ES : 1);
    const int64_t nseg = (L.D + seg_cols - 1) / seg_cols;
    const int64_t blocks = (runs * nseg + 7) / 8;
    if (vec)
        launch(scatter_runs<DT, true>, grid_for((const void*)scatter_runs<DT, true>, 256, blocks), 256, 0, s, L, P, nseg);
    else
        launch(scatter_runs<DT, false>, grid_for((const void*)scatter_runs<DT, false>, 256, blocks), 256, 0, s, L, P,
                                                                                                       nseg);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

template <int DT>
static psg_status launch_owner(const ScatterLaunch& L, cudaStream_t s)
{
    constexpr int ES = SV<DT>::ES;
    const bool pair = (DT == PSG_BF16 || DT == PSG_F16) && L.upd_cs == 1 && ((uintptr_t)L.upd + (uint64_t)L.upd_offset * ES) % 4 == 0 &&
                      ((uint64_t)L.upd_rs * ES) % 4 == 0;
    const int64_t chunk = OWNER_THREADS * (pair ? 2 : 1);
    const int64_t ncb = (L.D + chunk - 1) / chunk;
    if (ncb == 0) return PSG_OK;
    const size_t smem = (size_t)L.n * 4;
    const void* fn = pair ? (const void*)scatter_owner<DT, true> : (const void*)scatter_owner<DT, false>;
    if (set_max_dynamic_smem(fn, (int)kScatterPlanMaxN * 4) != cudaSuccess) return PSG_E_CUDA;
    const unsigned blocks = (unsigned)(L.V * ncb);
    const int idx16 = ((uintptr_t)L.idx % 16) == 0 ? 1 : 0;
    if (pair) launch(scatter_owner<DT, true>, blocks, OWNER_THREADS, smem, s, L, ncb, idx16);
    else launch(scatter_owner<DT, false>, blocks, OWNER_THREADS, smem, s, L, ncb, idx16);
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

psg_status launch_scatter(const ScatterLaunch& L, unsigned long long* keys, void* stream)
{
    if (L.n == 0) return PSG_OK;
    cudaStream_t s = (cudaStream_t)stream;
    if (L.n <= kScatterPlanMaxN && L.V <= OWNER_MAX_V && L.V * L.n <= OWNER_MAX_VN) {
        switch (L.dtype) {
        case PSG_F32: return launch_owner<PSG_F32>(L, s);
        case PSG_BF16: return launch_owner<PSG_BF16>(L, s);
        case PSG_F16: return launch_owner<PSG_F16>(L, s);
        case PSG_F64: return launch_owner<PSG_F64>(L, s);
        case PSG_I16: return launch_owner<PSG_I16>(L, s);
        case PSG_I8: return launch_owner<PSG_I8>(L, s);
        default: return launch_owner<PSG_I32>(L, s);
        }
    }
    if (L.n <= kScatterPlanMaxN && L.V < (int64_t(1) << 31) - 1) {
        switch (L.dtype) {
        case PSG_F32: return launch_planned<PSG_F32>(L, keys, s);
        case PSG_BF16: return launch_planned<PSG_BF16>(L, keys, s);
        case PSG_F16: return launch_planned<PSG_F16>(L, keys, s);
        case PSG_F64: return launch_planned<PSG_F64>(L, keys, s);
        case PSG_I16: return launch_planned<PSG_I16>(L, keys, s);
        case PSG_I8: return launch_planned<PSG_I8>(L, keys, s);
        default: return launch_planned<PSG_I32>(L, keys, s);
        }
    }
    // longer lists: 64-bit keys (idx << 32 | n) through a bitonic network
    const int64_t np2 = scatter_npow2(L.n);
    launch(make_keys, grid_for((const void*)make_keys, 256, (np2 + 255) / 256), 256, 0, s, L.idx, L.n, L.V, np2, keys,
                                                                                     L.status);
    const int64_t tiles = (np2 + LOCAL_SORT - 1) / LOCAL_SORT;
    launch(bitonic_local, (unsigned)tiles, 1024, 0, s, keys, np2, 0);
    for (int64_t k = 2 * LOCAL_SORT; k <= np2; k <<= 1) {
        for (int64_t j = k >> 1; j >= LOCAL_SORT; j >>= 1)
            launch(bitonic_global, grid_for((const void*)bitonic_global, 256, (np2 / 2 + 255) / 256), 256, 0, s, keys, np2, k, j);
        launch(bitonic_local, (unsigned)tiles, 1024, 0, s, keys, np2, k);
    }
    switch (L.dtype) {
    case PSG_F32: launch_accumulate<PSG_F32>(L, keys, s); break;
    case PSG_BF16: launch_accumulate<PSG_BF16>(L, keys, s); break;
    case PSG_F16: launch_accumulate<PSG_F16>(L, keys, s); break;
    case PSG_F64: launch_accumulate<PSG_F64>(L, keys, s); break;
    case PSG_I16: launch_accumulate<PSG_I16>(L, keys, s); break;
    case PSG_I8: launch_accumulate<PSG_I8>(L, keys, s); break;
    default: launch_accumulate<PSG_I32>(L, keys, s); break;
    }
    return cudaGetLastError() == cudaSuccess ? PSG_OK : PSG_E_CUDA;
}

}  // namespace psg
