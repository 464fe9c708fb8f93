// Row reduction skeleton (runtime-specialised per set of stage programs).
//
// A team of T = 1 << team_log2 threads (T <= 256, the block size) owns one
// row of length N (the last dim; limn, "Reading the schedule": a reduce is a
// cut and elementwise work fuses into it).  Each thread holds chunks lane,
// lane+T, ... of PSG_VEC cells.  When the row fits (kCH chunks per thread,
// kCH > 0) the inputs are loaded once into registers and every stage and the
// epilogue read them from there, so the row costs one HBM read and one
// write; otherwise every stage streams the row again.  A stage folds its prologue values per thread, then
// across the warp with shuffles and across the team's warps through shared
// memory in a fixed order (the same bits every run).  The running total is
// float32 (int32 for ints) and rounds into the stage dtype once (limn, "The
// op set": a reduce keeps its running total in float32).
//
// The including source defines kNin, kInMode[], kInDt[], kOutDt, kNstages,
// kStageOp[], kStageDt[], kCH, kPerRow, StageBody<S> and Epi.

template <int V> struct IC { static constexpr int value = V; };
template <int J, int N, class F>
__device__ __forceinline__ void sfor(F& f)
{
    if constexpr (J < N) {
        f(IC<J>{});
        sfor<J + 1, N>(f);
    }
}

#define PSG_RED_SUM 0
#define PSG_RED_MAX 1
constexpr int kNinP = kNin > 0 ? kNin : 1;
constexpr int kCHP = kCH > 0 ? kCH : 1;

// MAX: NaN propagates, +0 beats -0 on a tie, so any order gives the same bits
__device__ __forceinline__ float fmax_step(float acc, float x)
{
    if (acc != acc) return acc;
    if (x != x || x > acc || (x == acc && (__float_as_uint(x) >> 31) == 0)) return x;
    return acc;
}

template <int OP, int DT>
struct Fold {
    typedef typename VT<DT>::T T;
    static __device__ __forceinline__ T identity()
    {
        if constexpr (OP == PSG_RED_SUM) return (T)0;
        else if constexpr (DT == PSG_DT_I32) return (int)0x80000000;
        else if constexpr (DT == PSG_DT_I16) return -32768;
        else if constexpr (DT == PSG_DT_I8) return -128;
        else return __uint_as_float(0xff800000u);  // -inf
    }
    static __device__ __forceinline__ T step(T acc, T x)
    {
        if constexpr (OP == PSG_RED_SUM) {
            if constexpr (DT == PSG_DT_I32 || DT == PSG_DT_I16 || DT == PSG_DT_I8) return addi(acc, x);
            else return __fadd_rn(acc, x);
        } else {
            if constexpr (DT == PSG_DT_I32 || DT == PSG_DT_I16 || DT == PSG_DT_I8) return x > acc ? x : acc;
            else return fmax_step(acc, x);
        }
    }
    // the total rounds into the stage dtype once
    static __device__ __forceinline__ T finish(T v)
    {
        if constexpr (DT == PSG_DT_BF16) return rbf(v);
        else if constexpr (DT == PSG_DT_F16) return rh(v);
        else if constexpr (DT == PSG_DT_I16) return w16(v);
        else if constexpr (DT == PSG_DT_I8) return w8(v);
        else return v;
    }
};

__device__ __forceinline__ u32 as_bits(float x) { return __float_as_uint(x); }
__device__ __forceinline__ u32 as_bits(int x) { return (u32)x; }
template <class T> __device__ __forceinline__ T from_bits(u32 b);
template <> __device__ __forceinline__ float from_bits<float>(u32 b) { return __uint_as_float(b); }
template <> __device__ __forceinline__ int from_bits<int>(u32 b) { return (int)b; }

struct RedCtx {
    const PsgRedParams& p;
    const i64 (&roff)[kNinP];
    const bool (&rok)[kNinP];
    const u32 (&cache)[kNinP][kCHP][PSG_VEC];
    const u32 (&red)[PSG_MAXSTAGES];
    i64 col0;
    int nvalid;
    int j;  // chunk slot (compile-time after unrolling)
    template <int K>
    __device__ __forceinline__ void ldv(typename VT<kInDt[K]>::T (&d)[PSG_VEC]) const
    {
        typedef typename VT<kInDt[K]>::T T;
        if constexpr (kCH > 0 && kInMode[K] != PSG_M_UNIFORM) {
#pragma unroll
            for (int v = 0; v < PSG_VEC; ++v) d[v] = from_bits<T>(cache[K][j][v]);
        } else {
            ld_chunk<kInDt[K], kInMode[K]>(p.in[K], roff[K], rok[K], col0, nvalid, d);
        }
    }
    template <int K>
    __device__ __forceinline__ typename VT<kInDt[K]>::T ld1() const
    {
        return ld_first<kInDt[K], kInMode[K]>(p.in[K], roff[K], rok[K], col0);
    }
    __device__ __forceinline__ float redf(int s) const { return __uint_as_float(red[s]); }
    __device__ __forceinline__ int redi(int s) const { return (int)red[s]; }
};

// fold v across the team (threads [team*T, team*T + T) of the block)
template <int OP, int DT>
__device__ __forceinline__ typename VT<DT>::T team_fold(typename VT<DT>::T v, int team_log2, u32* sm)
{
    typedef Fold<OP, DT> F;
    const int T = 1 << team_log2;
    const int width = T < 32 ? T : 32;
    for (int off = width >> 1; off > 0; off >>= 1) {
        const u32 o = __shfl_xor_sync(0xffffffffu, as_bits(v), off, 32);
        v = F::step(v, from_bits<typename VT<DT>::T>(o));
    }
    if (T > 32) {
        const int warp = threadIdx.x >> 5;
        const int W = T >> 5;
        const int team = threadIdx.x >> team_log2;
        if ((threadIdx.x & 31) == 0) sm[warp] = as_bits(v);
        __syncthreads();
        v = from_bits<typename VT<DT>::T>(sm[team * W]);
        for (int w = 1; w < W; ++w) v = F::step(v, from_bits<typename VT<DT>::T>(sm[team * W + w]));
        __syncthreads();
    }
    return v;
}

extern "C" __global__ void __launch_bounds__(256) psg_reduce(const __grid_constant__ PsgRedParams p)
{
    __shared__ u32 sm[32];
    const int T = 1 << p.team_log2;
    const int teams = blockDim.x >> p.team_log2;
    const int team = threadIdx.x >> p.team_log2;
    const int lane = threadIdx.x & (T - 1);
    // every team of the block runs the same number of iterations, so the
    // barriers inside team_fold are reached by all threads
    for (i64 base = (i64)blockIdx.x * teams; base < p.rows; base += (i64)gridDim.x * teams) {
        const i64 row = base + team;
        const bool active = row < p.rows;
        i64 roff[kNinP];
        bool rok[kNinP];
        i64 ooff = 0;
        if (active) {
            PsgOperand outp = p.out;
            row_offsets<kNin>(p.in, outp, p.shape, p.nd, row, roff, rok, kInMode, ooff);
        } else {
#pragma unroll
            for (int k = 0; k < kNinP; ++k) { roff[k] = 0; rok[k] = false; }
        }
        // load the row once when it fits in registers
        u32 cache[kNinP][kCHP][PSG_VEC];
        if constexpr (kCH > 0) {
#pragma unroll
            for (int j = 0; j < kCH; ++j) {
                const i64 ch = lane + (i64)j * T;
                const i64 col0 = ch * PSG_VEC;
                const i64 left = p.inner - col0;
                const int nvalid = !active || left <= 0 ? 0 : left < PSG_VEC ? (int)left : PSG_VEC;
                auto ldk = [&](auto kt) {
                    constexpr int K = decltype(kt)::value;
                    if constexpr (kInMode[K] != PSG_M_UNIFORM) {
                        typename VT<kInDt[K]>::T d[PSG_VEC];
                        if (nvalid > 0) ld_chunk<kInDt[K], kInMode[K]>(p.in[K], roff[K], rok[K], col0, nvalid, d);
#pragma unroll
                        for (int v = 0; v < PSG_VEC; ++v) cache[K][j][v] = nvalid > 0 ? as_bits(d[v]) : 0u;
                    }
                };
                sfor<0, kNin>(ldk);
            }
        }
        u32 red[PSG_MAXSTAGES] = {0u, 0u, 0u, 0u};
        auto stage = [&](auto st) {
            constexpr int S = decltype(st)::value;
            constexpr int OP = kStageOp[S];
            constexpr int DT = kStageDt[S];
            typedef Fold<OP, DT> F;
            typename VT<DT>::T acc = F::identity();
            const int nch = kCH > 0 ? kCH : (int)((p.chunks - lane + T - 1) / T);
#pragma unroll
            for (int j = 0; j < (kCH > 0 ? kCH : 1); ++j) {
                for (int jj = (kCH > 0 ? j : 0); jj < (kCH > 0 ? j + 1 : nch); ++jj) {
                    const i64 ch = lane + (i64)jj * T;
                    const i64 col0 = ch * PSG_VEC;
                    const i64 left = p.inner - col0;
                    if (!active || left <= 0) continue;
                    const int nvalid = left < PSG_VEC ? (int)left : PSG_VEC;
                    const RedCtx c{p, roff, rok, cache, red, col0, nvalid, j};
                    typename VT<DT>::T y[PSG_VEC];
                    StageBody<S>::eval(c, y);
#pragma unroll
                    for (int v = 0; v < PSG_VEC; ++v)
                        if (v < nvalid) acc = F::step(acc, y[v]);
                }
            }
            acc = team_fold<OP, DT>(acc, p.team_log2, sm);
            red[S] = as_bits(F::finish(acc));
        };
        sfor<0, kNstages>(stage);
        if (!active) continue;
        if constexpr (kPerRow) {
            if (lane == 0) {
                const RedCtx c{p, roff, rok, cache, red, 0, 1, 0};
                typename VT<kOutDt>::T y[PSG_VEC];
                Epi::eval(c, y);
                st_cell<kOutDt>((void*)p.out.ptr, ooff, y[0]);
            }
        } else {
            const int nch = kCH > 0 ? kCH : (int)((p.chunks - lane + T - 1) / T);
#pragma unroll
            for (int j = 0; j < (kCH > 0 ? kCH : 1); ++j) {
                for (int jj = (kCH > 0 ? j : 0); jj < (kCH > 0 ? j + 1 : nch); ++jj) {
                    const i64 ch = lane + (i64)jj * T;
                    const i64 col0 = ch * PSG_VEC;
                    const i64 left = p.inner - col0;
                    if (left <= 0) continue;
                    const int nvalid = left < PSG_VEC ? (int)left : PSG_VEC;
                    const RedCtx c{p, roff, rok, cache, red, col0, nvalid, j};
                    typename VT<kOutDt>::T y[PSG_VEC];
                    Epi::eval(c, y);
                    st_chunk<kOutDt>(p.out, ooff, col0, nvalid, y);
                }
            }
        }
    }
}
